"""ctypes binding of libpagedkv.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
turns torch tensors into device pointers, passes the current CUDA stream and
raises on a non-OK status.  If the library is missing it raises: there is no
fallback path.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pagedkv.h")

KV_BF16, KV_FP8_E4M3 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "workspace missing or too small",
          4: "CUDA error", 5: "device-side index or length error", 6: "device-side wait timed out",
          7: "no free cache block and none evictable", 8: "unknown (or already registered) sequence id"}
DEVERR_BLOCK_ID, DEVERR_LENGTH, DEVERR_SLOT, DEVERR_TIMEOUT, DEVERR_RANGE = 1, 2, 4, 8, 16

_lock = threading.Lock()
_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, 'unknown')} (status {status})")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p)]


def lib():
    """Load libpagedkv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libpagedkv.so not found at {LIB_PATH}: build it first "
                                   "(`python -m paged_kv_decode_14_gb300.build`)")
            L = ctypes.CDLL(LIB_PATH)
            c = ctypes
            vp, i32, i64 = c.c_void_p, c.c_int32, c.c_int64
            L.pkv_paged_kv_append.restype = c.c_int
            L.pkv_paged_kv_append.argtypes = [c.POINTER(CacheDesc), vp, vp, vp, i64, vp, vp]
            L.pkv_attention_workspace_size.restype = c.c_size_t
            L.pkv_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
            L.pkv_workspace_init.restype = c.c_int
            L.pkv_workspace_init.argtypes = [vp, c.c_size_t, vp]
            L.pkv_paged_attention.restype = c.c_int
            L.pkv_paged_attention.argtypes = [c.POINTER(CacheDesc), vp, i32, vp, i32, vp, vp, i32, i32,
                                              c.c_float, vp, vp, c.c_size_t, i32, vp]
            L.pkv_paged_attention_noalloc.restype = c.c_int
            L.pkv_paged_attention_noalloc.argtypes = [c.POINTER(CacheDesc), vp, i32, vp, i32, vp, vp, i32, i32,
                                                      c.c_float, vp, i32, vp, vp]
            L.pkv_paged_prefill.restype = c.c_int
            L.pkv_paged_prefill.argtypes = [c.POINTER(CacheDesc), vp, i32, vp, i32, vp, vp, i32, i32, c.c_float, vp,
                                            vp, vp]
            L.pkv_kvmgr_create.restype = vp
            L.pkv_kvmgr_create.argtypes = [i64]
            L.pkv_kvmgr_destroy.restype = None
            L.pkv_kvmgr_destroy.argtypes = [vp]
            L.pkv_kvmgr_add_sequence.restype = c.c_int
            L.pkv_kvmgr_add_sequence.argtypes = [vp, i64, vp, i64, c.POINTER(i64), vp]
            L.pkv_kvmgr_append.restype = c.c_int
            L.pkv_kvmgr_append.argtypes = [vp, i64, vp, i64, vp, vp, c.POINTER(i32)]
            for nm in ("pkv_kvmgr_commit", "pkv_kvmgr_release"):
                getattr(L, nm).restype = c.c_int
                getattr(L, nm).argtypes = [vp, i64]
            L.pkv_kvmgr_fork.restype = c.c_int
            L.pkv_kvmgr_fork.argtypes = [vp, i64, i64]
            L.pkv_kvmgr_tables.restype = c.c_int
            L.pkv_kvmgr_tables.argtypes = [vp, vp, i32, i32, vp, vp]
            L.pkv_kvmgr_num_free.restype = i64
            L.pkv_kvmgr_num_free.argtypes = [vp]
            L.pkv_kvmgr_num_cached.restype = i64
            L.pkv_kvmgr_num_cached.argtypes = [vp]
            L.pkv_kvmgr_refcount.restype = i32
            L.pkv_kvmgr_refcount.argtypes = [vp, i32]
            L.pkv_cascade_workspace_size.restype = c.c_size_t
            L.pkv_cascade_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            L.pkv_paged_attention_cascade.restype = c.c_int
            L.pkv_paged_attention_cascade.argtypes = [c.POINTER(CacheDesc), vp, i32, vp, i32, vp, vp, i32, i32, vp, vp,
                                                      i32, i32, c.c_float, vp, vp, c.c_size_t, vp]
            L.pkv_paged_kv_append_rope.restype = c.c_int
            L.pkv_paged_kv_append_rope.argtypes = [c.POINTER(CacheDesc), vp, vp, vp, i64, vp, c.c_float, vp, i32,
                                                   i32, vp, vp]
            L.pkv_copy_blocks.restype = c.c_int
            L.pkv_copy_blocks.argtypes = [c.POINTER(CacheDesc), vp, i32, vp, vp, vp]
            L.pkv_debug_set_wait_limit.restype = None
            L.pkv_debug_set_wait_limit.argtypes = [c.c_uint64, vp]
            L.pkv_read_device_error.restype = c.c_int
            L.pkv_read_device_error.argtypes = [vp, c.POINTER(i32), vp]
            L.pkv_status_string.restype = c.c_char_p
            L.pkv_status_string.argtypes = [c.c_int]
            L.pkv_version.restype = c.c_char_p
            L.pkv_version.argtypes = []
            _lib = L
    return _lib


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class PagedKVCache:
    """A paged K/V cache in the library's layout: two device buffers of
    [num_blocks][num_kv_heads][16 * head_dim] elements (bf16 or e4m3 bytes),
    plus the per-(block, kv-head) fp32 scales of an FP8 cache."""

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, kv_dtype: str = "bf16",
                 device="cuda", k=None, v=None, k_scales=None, v_scales=None):
        self.num_blocks, self.num_kv_heads, self.head_dim = num_blocks, num_kv_heads, head_dim
        self.kv_dtype = kv_dtype
        tdt = torch.uint8 if kv_dtype == "fp8" else torch.bfloat16
        shape = (num_blocks, num_kv_heads, 16 * head_dim)
        self.k = k if k is not None else torch.empty(shape, dtype=tdt, device=device)
        self.v = v if v is not None else torch.empty(shape, dtype=tdt, device=device)
        self.k_scales, self.v_scales = k_scales, v_scales
        if kv_dtype == "fp8" and (k_scales is None or v_scales is None):
            raise ValueError("an FP8 cache needs k_scales and v_scales")

    def desc(self) -> CacheDesc:
        for t in (self.k, self.v):
            if not t.is_contiguous():
                raise ValueError("cache buffers must be contiguous")
        for t in (self.k_scales, self.v_scales):
            if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
                raise ValueError("scales must be contiguous float32")
        return CacheDesc(self.num_blocks, 16, self.num_kv_heads, self.head_dim,
                         KV_FP8_E4M3 if self.kv_dtype == "fp8" else KV_BF16,
                         self.k.data_ptr(), self.v.data_ptr(),
                         None if self.k_scales is None else self.k_scales.data_ptr(),
                         None if self.v_scales is None else self.v_scales.data_ptr())


def _check(st: int, what: str):
    if st != 0:
        raise PagedKVError(st, what)


def append(cache: PagedKVCache, k_new, v_new, slot_mapping, device_error=None, stream=None):
    """pkv_paged_kv_append: k_new/v_new bf16 [T, Hkv, D], slot_mapping int64 [T]."""
    for t in (k_new, v_new):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("k_new / v_new must be contiguous bfloat16")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    d = cache.desc()
    st = lib().pkv_paged_kv_append(ctypes.byref(d), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                   int(slot_mapping.numel()), _ptr(device_error), _stream(stream))
    _check(st, "pkv_paged_kv_append")


def append_rope(cache: PagedKVCache, k_new, v_new, slot_mapping, positions=None, theta: float = 10000.0, q=None,
                fp8_scales_from_values: bool = False, device_error=None, stream=None):
    """pkv_paged_kv_append_rope: append with K rotated at `positions` (int32
    [T], None = no rotation), q rows [T, Hq, D] rotated in place, and
    optionally the FP8 scales of the blocks this call starts chosen from the
    values (written into cache.k_scales / v_scales)."""
    for t in (k_new, v_new):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("k_new / v_new must be contiguous bfloat16")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if positions is not None and (positions.dtype != torch.int32 or not positions.is_contiguous()):
        raise ValueError("positions must be contiguous int32")
    if q is not None and (q.dtype != torch.bfloat16 or not q.is_contiguous()):
        raise ValueError("q must be contiguous bfloat16")
    d = cache.desc()
    st = lib().pkv_paged_kv_append_rope(ctypes.byref(d), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                        int(slot_mapping.numel()), _ptr(positions), float(theta), _ptr(q),
                                        int(q.shape[1]) if q is not None else 0, int(bool(fp8_scales_from_values)),
                                        _ptr(device_error), _stream(stream))
    _check(st, "pkv_paged_kv_append_rope")


def workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_q_len, num_ctas=0) -> int:
    n = lib().pkv_attention_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_q_len, num_ctas)
    if n == 0:
        raise PagedKVError(1, "pkv_attention_workspace_size")
    return int(n)


def make_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_q_len, num_ctas=0, device="cuda",
                   stream=None):
    n = workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_q_len, num_ctas)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(lib().pkv_workspace_init(_ptr(ws), n, _stream(stream)), "pkv_workspace_init")
    return ws


def workspace_init(workspace, stream=None):
    """pkv_workspace_init: zero a workspace (needed once, and after a timeout)."""
    _check(lib().pkv_workspace_init(_ptr(workspace), int(workspace.numel()), _stream(stream)), "pkv_workspace_init")


def attention(cache: PagedKVCache, q, block_tables, context_lens, q_lens, max_q_len: int, scale: float,
              workspace, out=None, num_ctas: int = 0, stream=None):
    """pkv_paged_attention: q bf16 [sum q_lens, Hq, D] -> out bf16 of the same shape."""
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be contiguous bfloat16 [rows, Hq, D]")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"), (q_lens, "q_lens")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    if out is None:
        out = torch.empty_like(q)
    d = cache.desc()
    st = lib().pkv_paged_attention(ctypes.byref(d), _ptr(q), int(q.shape[1]), _ptr(block_tables),
                                   int(block_tables.shape[1]), _ptr(context_lens), _ptr(q_lens),
                                   int(context_lens.numel()), int(max_q_len), float(scale), _ptr(out),
                                   _ptr(workspace), int(workspace.numel()), int(num_ctas), _stream(stream))
    _check(st, "pkv_paged_attention")
    return out


def make_cascade_workspace(num_seqs, num_groups, num_q_heads, num_kv_heads, head_dim, max_q_len, max_group_q_len,
                           device="cuda", stream=None):
    n = lib().pkv_cascade_workspace_size(num_seqs, num_groups, num_q_heads, num_kv_heads, head_dim, max_q_len,
                                         max_group_q_len)
    if n == 0:
        raise PagedKVError(1, "pkv_cascade_workspace_size")
    ws = torch.empty(int(n), dtype=torch.uint8, device=device)
    _check(lib().pkv_workspace_init(_ptr(ws), int(n), _stream(stream)), "pkv_workspace_init")
    return ws


def attention_cascade(cache: PagedKVCache, q, block_tables, context_lens, q_lens, max_q_len: int, group_starts,
                      group_prefix_lens, max_group_q_len: int, scale: float, workspace, out=None, stream=None):
    """pkv_paged_attention_cascade: attention with each group's shared prefix
    attended once for the whole group (group_starts int32 [G + 1],
    group_prefix_lens int32 [G], device)."""
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be contiguous bfloat16 [rows, Hq, D]")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"), (q_lens, "q_lens"),
                    (group_starts, "group_starts"), (group_prefix_lens, "group_prefix_lens")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    if out is None:
        out = torch.empty_like(q)
    d = cache.desc()
    st = lib().pkv_paged_attention_cascade(ctypes.byref(d), _ptr(q), int(q.shape[1]), _ptr(block_tables),
                                           int(block_tables.shape[1]), _ptr(context_lens), _ptr(q_lens),
                                           int(context_lens.numel()), int(max_q_len), _ptr(group_starts),
                                           _ptr(group_prefix_lens), int(group_prefix_lens.numel()),
                                           int(max_group_q_len), float(scale), _ptr(out), _ptr(workspace),
                                           int(workspace.numel()), _stream(stream))
    _check(st, "pkv_paged_attention_cascade")
    return out


def attention_noalloc(cache: PagedKVCache, q, block_tables, context_lens, q_lens, max_q_len: int, scale: float,
                      out=None, num_ctas: int = 0, device_error=None, stream=None):
    """pkv_paged_attention_noalloc: like attention(), with the library's static
    scratch array instead of a caller workspace (for callers that cannot
    allocate device memory).  Calls that overlap on the GPU race."""
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be contiguous bfloat16 [rows, Hq, D]")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"), (q_lens, "q_lens")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    if out is None:
        out = torch.empty_like(q)
    d = cache.desc()
    st = lib().pkv_paged_attention_noalloc(ctypes.byref(d), _ptr(q), int(q.shape[1]), _ptr(block_tables),
                                           int(block_tables.shape[1]), _ptr(context_lens), _ptr(q_lens),
                                           int(context_lens.numel()), int(max_q_len), float(scale), _ptr(out),
                                           int(num_ctas), _ptr(device_error), _stream(stream))
    _check(st, "pkv_paged_attention_noalloc")
    return out


def prefill(cache: PagedKVCache, q, block_tables, context_lens, q_lens, max_q_len: int, scale: float, out=None,
            device_error=None, stream=None):
    """pkv_paged_prefill: causal attention of long query windows (prompts or
    prompt chunks) on the tensor cores; q bf16 [sum q_lens, Hq, D] -> out of
    the same shape.  bf16 caches, Hq / Hkv dividing 128."""
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be contiguous bfloat16 [rows, Hq, D]")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"), (q_lens, "q_lens")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    if out is None:
        out = torch.empty_like(q)
    d = cache.desc()
    st = lib().pkv_paged_prefill(ctypes.byref(d), _ptr(q), int(q.shape[1]), _ptr(block_tables),
                                 int(block_tables.shape[1]), _ptr(context_lens), _ptr(q_lens),
                                 int(context_lens.numel()), int(max_q_len), float(scale), _ptr(out),
                                 _ptr(device_error), _stream(stream))
    _check(st, "pkv_paged_prefill")
    return out


def read_device_error(error_word, stream=None) -> int:
    """Read and clear a device error word (workspace or append flag); syncs."""
    code = ctypes.c_int32(0)
    st = lib().pkv_read_device_error(_ptr(error_word), ctypes.byref(code), _stream(stream))
    if st not in (0, 5, 6):
        _check(st, "pkv_read_device_error")
    return int(code.value)


class KVManager:
    """The library's host-side block manager (pkv_kvmgr_*): block allocation,
    reference counts, copy-on-write and radix prefix reuse; it hands out the
    slots and block tables the append and attention calls take.  Host memory
    only (numpy arrays in and out)."""

    def __init__(self, num_blocks: int):
        self._lib = lib()
        self._h = self._lib.pkv_kvmgr_create(int(num_blocks))
        if not self._h:
            raise PagedKVError(1, "pkv_kvmgr_create")
        self.num_blocks = int(num_blocks)

    def close(self):
        if self._h:
            self._lib.pkv_kvmgr_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _i32(a):
        import numpy as np
        return np.ascontiguousarray(a, dtype=np.int32)

    def add_sequence(self, seq: int, tokens):
        """-> (cached_tokens, slots of the other prompt tokens: int64 array)."""
        import numpy as np
        t = self._i32(tokens)
        slots = np.zeros(len(t), dtype=np.int64)
        cached = ctypes.c_int64(0)
        _check(self._lib.pkv_kvmgr_add_sequence(self._h, int(seq), t.ctypes.data, len(t), ctypes.byref(cached),
                                                slots.ctypes.data), "pkv_kvmgr_add_sequence")
        return int(cached.value), slots[:len(t) - int(cached.value)].copy()

    def append(self, seq: int, tokens):
        """-> (slots: int64 array, copy-on-write pair (src, dst) or None)."""
        import numpy as np
        t = self._i32(tokens)
        slots = np.zeros(len(t), dtype=np.int64)
        copy = np.zeros(2, dtype=np.int32)
        ncopy = ctypes.c_int32(0)
        _check(self._lib.pkv_kvmgr_append(self._h, int(seq), t.ctypes.data, len(t), slots.ctypes.data,
                                          copy.ctypes.data, ctypes.byref(ncopy)), "pkv_kvmgr_append")
        return slots, (int(copy[0]), int(copy[1])) if ncopy.value else None

    def commit(self, seq: int):
        _check(self._lib.pkv_kvmgr_commit(self._h, int(seq)), "pkv_kvmgr_commit")

    def fork(self, parent: int, child: int):
        _check(self._lib.pkv_kvmgr_fork(self._h, int(parent), int(child)), "pkv_kvmgr_fork")

    def release(self, seq: int):
        _check(self._lib.pkv_kvmgr_release(self._h, int(seq)), "pkv_kvmgr_release")

    def tables(self, seqs, max_blocks: int):
        """-> (block_tables int32 [n, max_blocks] (-1 padded), context_lens int32 [n])."""
        import numpy as np
        s = np.ascontiguousarray(seqs, dtype=np.int64)
        bt = np.zeros((len(s), max_blocks), dtype=np.int32)
        lens = np.zeros(len(s), dtype=np.int32)
        _check(self._lib.pkv_kvmgr_tables(self._h, s.ctypes.data, len(s), int(max_blocks), bt.ctypes.data,
                                          lens.ctypes.data), "pkv_kvmgr_tables")
        return bt, lens

    def num_free(self) -> int:
        return int(self._lib.pkv_kvmgr_num_free(self._h))

    def num_cached(self) -> int:
        return int(self._lib.pkv_kvmgr_num_cached(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_kvmgr_refcount(self._h, int(block)))


def copy_blocks(cache: PagedKVCache, pairs, stream=None):
    """pkv_copy_blocks: device int32 [n, 2] (src, dst) block pairs; an FP8
    cache's scales are copied too."""
    if pairs.dtype != torch.int32 or not pairs.is_contiguous():
        raise ValueError("pairs must be contiguous int32 [n, 2]")
    d = cache.desc()
    fp8 = cache.kv_dtype == "fp8"
    _check(lib().pkv_copy_blocks(ctypes.byref(d), _ptr(pairs), int(pairs.shape[0]),
                                 _ptr(cache.k_scales) if fp8 else None, _ptr(cache.v_scales) if fp8 else None,
                                 _stream(stream)), "pkv_copy_blocks")


def debug_set_wait_limit(limit_ns: int = 0, hold_flag=None):
    """Test hook of the timeout path (pkv_debug_set_wait_limit): the wait
    limit of later attention launches (0 = the default 2 s) and an optional
    device int32 flag the kernel waits on before its first K/V copy."""
    lib().pkv_debug_set_wait_limit(int(limit_ns), _ptr(hold_flag))


def version() -> str:
    return lib().pkv_version().decode()

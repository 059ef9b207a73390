"""ctypes wrapper around the plain C fp64 oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg may use this module; the library's product path
never does.  It shares no code with the CUDA library.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16, KV_FP8 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
                               "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            c = ctypes
            L.oracle_e4m3_decode.restype = c.c_double
            L.oracle_e4m3_decode.argtypes = [c.c_uint8]
            L.oracle_e4m3_encode.restype = c.c_uint8
            L.oracle_e4m3_encode.argtypes = [c.c_float]
            L.oracle_bf16_round.restype = c.c_uint16
            L.oracle_bf16_round.argtypes = [c.c_double]
            L.oracle_cache_index.restype = c.c_size_t
            L.oracle_cache_index.argtypes = [c.c_int64, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int]
            L.oracle_paged_kv_append.restype = c.c_int64
            L.oracle_paged_kv_append.argtypes = [c.c_int, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,
                                                 c.c_int64, c.c_int, c.c_int, c.c_void_p, c.c_void_p,
                                                 c.c_void_p, c.c_int64]
            L.oracle_paged_attention.restype = c.c_int
            L.oracle_paged_attention.argtypes = [c.c_int, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,
                                                 c.c_int64, c.c_int, c.c_int, c.c_void_p, c.c_int,
                                                 c.c_void_p, c.c_int, c.c_void_p, c.c_void_p, c.c_int,
                                                 c.c_float, c.c_void_p, c.c_void_p, c.c_int]
            L.oracle_rope.restype = None
            L.oracle_rope.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_int, c.c_int, c.c_double]
            L.oracle_fp8_autoscale.restype = None
            L.oracle_fp8_autoscale.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_int, c.c_int,
                                               c.c_int64, c.c_void_p, c.c_void_p]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    return lib().oracle_e4m3_encode(float(x))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    f = lib().oracle_e4m3_encode
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.fromiter((f(float(v)) for v in flat), dtype=np.uint8, count=flat.size).reshape(np.shape(x))


def bf16_round(x: float) -> int:
    return lib().oracle_bf16_round(float(x))


def cache_index(blk, g, off, d, num_kv_heads, head_dim, elem_bytes) -> int:
    return lib().oracle_cache_index(blk, g, off, d, num_kv_heads, head_dim, elem_bytes)


def paged_kv_append(kv_dtype, k_cache, v_cache, k_scales, v_scales, num_blocks, num_kv_heads,
                    head_dim, k_new, v_new, slots) -> int:
    """In-place append into numpy cache buffers; returns the number of skipped
    out-of-range slots."""
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    ks = None if k_scales is None else np.ascontiguousarray(k_scales, dtype=np.float32)
    vs = None if v_scales is None else np.ascontiguousarray(v_scales, dtype=np.float32)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    r = lib().oracle_paged_kv_append(kv_dtype, _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs),
                                     num_blocks, num_kv_heads, head_dim, _ptr(k_new), _ptr(v_new),
                                     _ptr(slots), slots.shape[0])
    if r < 0:
        raise ValueError("oracle append: bad arguments")
    return r


def paged_attention(kv_dtype, k_cache, v_cache, k_scales, v_scales, num_blocks, num_kv_heads,
                    head_dim, q, num_q_heads, block_tables, context_lens, q_lens, scale,
                    nthreads: int | None = None):
    """Returns (out fp64, out bf16 bits), both [sum q_lens, Hq, D]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    ks = None if k_scales is None else np.ascontiguousarray(k_scales, dtype=np.float32)
    vs = None if v_scales is None else np.ascontiguousarray(v_scales, dtype=np.float32)
    rows = int(ql.sum())
    out = np.zeros((rows, num_q_heads, head_dim), dtype=np.float64)
    outb = np.zeros((rows, num_q_heads, head_dim), dtype=np.uint16)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    mb = bt.shape[1] if bt.ndim == 2 else 1
    st = lib().oracle_paged_attention(kv_dtype, _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs),
                                      num_blocks, num_kv_heads, head_dim, _ptr(q), num_q_heads,
                                      _ptr(bt), mb, _ptr(cl), _ptr(ql), cl.shape[0], float(scale),
                                      _ptr(out), _ptr(outb), int(nthreads))
    if st != 0:
        raise ValueError(f"oracle attention failed with status {st}")
    return out, outb


def rope(x, positions, theta: float) -> np.ndarray:
    """Rotate-half RoPE of bf16 rows x [T, H, D] at positions [T], fp64 then
    bf16 RNE (oracle_rope)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    y = np.empty_like(x)
    T, H, D = x.shape
    lib().oracle_rope(_ptr(x), _ptr(y), _ptr(pos), T, H, D, float(theta))
    return y


def fp8_autoscale(k_new, v_new, slots, num_blocks, k_scales, v_scales):
    """In-place: the scales of the blocks this append starts, from its values
    (oracle_fp8_autoscale)."""
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    assert k_scales.flags.c_contiguous and v_scales.flags.c_contiguous
    T, Hkv, D = k_new.shape
    lib().oracle_fp8_autoscale(_ptr(k_new), _ptr(v_new), _ptr(slots), T, Hkv, D, int(num_blocks),
                               _ptr(k_scales), _ptr(v_scales))


# ---------------------------------------------------------------- workload helpers

def build_cache(w, with_step: bool = True):
    """Build the resident cache of a workload with the oracle's own append:
    prefill tokens, then (optionally) the step's new tokens."""
    kd = KV_FP8 if w.kv_dtype == "fp8" else KV_BF16
    kc, vc = w.empty_cache(), w.empty_cache()
    paged_kv_append(kd, kc, vc, w.k_scales, w.v_scales, w.num_blocks, w.num_kv_heads, w.head_dim,
                    w.prefill_k, w.prefill_v, w.prefill_slots)
    if with_step:
        paged_kv_append(kd, kc, vc, w.k_scales, w.v_scales, w.num_blocks, w.num_kv_heads, w.head_dim,
                        w.k_new, w.v_new, w.slots)
    return kc, vc


def attend(w, kc, vc, nthreads=None):
    kd = KV_FP8 if w.kv_dtype == "fp8" else KV_BF16
    return paged_attention(kd, kc, vc, w.k_scales, w.v_scales, w.num_blocks, w.num_kv_heads,
                           w.head_dim, w.q, w.num_q_heads, w.block_tables, w.context_lens,
                           w.q_lens, w.scale, nthreads)

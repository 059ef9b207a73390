"""Seeded synthetic workloads for paged-KV decode attention.

This module only draws inputs: random tensors, context lengths, block tables,
slot mappings and FP8 scales.  It holds none of the attention or append
arithmetic, so both the CUDA path and the CPU oracle can consume it.

Every workload is described the same way:

* ``prefill`` tokens: K/V source rows (bf16 bit patterns) plus the int64 slot
  each one is appended to before the timed step.  The resident cache is built
  by appending them, on each side with its own append.
* ``step``: the decode step itself -- ``q`` plus the new K/V rows and their
  slots (appended first, then attended: the context length of a sequence
  counts the tokens just appended).
* ``block_tables`` padded with -1, ``context_lens`` and ``q_lens`` (int32).

Value recipe (all configs): q/K/V ~ N(0, 1) drawn in fp32 and rounded to
bf16 (round to nearest even).  Physical blocks come from a seeded permutation
of the pool.  For the FP8 cache, each source element is multiplied by 8 with
probability 1 %, and the per-(block, kv-head) scale is absmax / 448 over the
source values that land in that block (1.0 if the block is empty or all zero).

The five named configurations follow the problem statement of the paged-KV
decode pages (inferd README "Paged KV" / lfm25-inference README "Paged
GQA/XQA Decode Attention"), with shapes and distributions of a continuous
decode batch, a multi-turn prefix-reuse batch, a speculative verify batch and
a long ragged FP8 batch.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
BF16_NAN = np.uint16(0x7FC0)
FP8_NAN = np.uint8(0x7F)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs only; no NaN)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str                    # "bf16" or "fp8"
    scale: float                     # softmax scale (fp32 value)
    num_blocks: int
    context_lens: np.ndarray         # [B] int32, includes the step's tokens
    q_lens: np.ndarray               # [B] int32
    block_tables: np.ndarray         # [B, MB] int32, -1 padded
    prefill_k: np.ndarray            # [Np, Hkv, D] uint16 (bf16 bits)
    prefill_v: np.ndarray
    prefill_slots: np.ndarray        # [Np] int64
    q: np.ndarray                    # [sum q_lens, Hq, D] uint16
    k_new: np.ndarray                # [sum q_lens, Hkv, D] uint16
    v_new: np.ndarray
    slots: np.ndarray                # [sum q_lens] int64
    k_scales: np.ndarray | None = None   # [NB, Hkv] float32 (fp8 only)
    v_scales: np.ndarray | None = None
    info: dict = field(default_factory=dict)

    @property
    def block_size(self) -> int:
        return BLOCK_SIZE

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "fp8" else 2

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    def cache_elems(self) -> int:
        return self.num_blocks * self.num_kv_heads * BLOCK_SIZE * self.head_dim

    def empty_cache(self) -> np.ndarray:
        """One cache buffer filled with the NaN sentinel (unused slots stay NaN)."""
        n = self.cache_elems()
        if self.kv_dtype == "fp8":
            return np.full(n, FP8_NAN, dtype=np.uint8)
        return np.full(n, BF16_NAN, dtype=np.uint16)

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one attention step reads (every resident token once
        per kv-head, K and V; FP8 adds two fp32 scales per block per kv-head)."""
        total_tokens = int(self.context_lens.astype(np.int64).sum())
        b = total_tokens * self.num_kv_heads * self.head_dim * 2 * self.elem_bytes
        if self.kv_dtype == "fp8":
            nblk = int(((self.context_lens.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE).sum())
            b += nblk * self.num_kv_heads * 2 * 4
        return b

    def unique_kv_bytes(self) -> int:
        """KV bytes counting each distinct physical block once (prefix sharing)."""
        used = set()
        for b in range(self.num_seqs):
            nb = (int(self.context_lens[b]) + BLOCK_SIZE - 1) // BLOCK_SIZE
            for j in range(nb):
                used.add(int(self.block_tables[b, j]))
        # a block's resident tokens: the largest fill any sequence reads from it
        fill = {}
        for b in range(self.num_seqs):
            L = int(self.context_lens[b])
            nb = (L + BLOCK_SIZE - 1) // BLOCK_SIZE
            for j in range(nb):
                blk = int(self.block_tables[b, j])
                fill[blk] = max(fill.get(blk, 0), min(BLOCK_SIZE, L - j * BLOCK_SIZE))
        toks = sum(fill.values())
        b = toks * self.num_kv_heads * self.head_dim * 2 * self.elem_bytes
        if self.kv_dtype == "fp8":
            b += len(used) * self.num_kv_heads * 2 * 4
        return b

    def prefix_groups(self):
        """(group_starts [G + 1], group_prefix_lens [G]) int32: the batch cut
        into consecutive groups, each a shared_prefix group or a sequence on
        its own (prefix 0)."""
        starts, plens, b = [0], [], 0
        groups = {first: (n, ptoks) for first, n, ptoks in self.info.get("shared_prefix", [])}
        while b < self.num_seqs:
            n, ptoks = groups.get(b, (1, 0))
            b += n
            starts.append(b)
            plens.append(ptoks)
        return np.asarray(starts, np.int32), np.asarray(plens, np.int32)

    def step_io_bytes(self) -> tuple[int, int]:
        """(host->device, device->host) bytes of one decode step's per-step inputs
        and output: q, new K/V, slots, block tables, lens in; out back."""
        hin = (self.q.nbytes + self.k_new.nbytes + self.v_new.nbytes + self.slots.nbytes
               + self.block_tables.nbytes + self.context_lens.nbytes + self.q_lens.nbytes)
        hout = self.q.nbytes
        return hin, hout


def _normal_bf16(rng: np.random.Generator, shape, outlier_p: float = 0.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if outlier_p > 0.0:
        mask = rng.random(size=shape, dtype=np.float32) < outlier_p
        x = np.where(mask, x * np.float32(8.0), x)
    return bf16_bits(x)


def _fp8_scales(num_blocks, Hkv, D, src_k, src_v, src_slots):
    """absmax / 448 per (block, kv-head) over the source rows stored there."""
    ks = np.zeros((num_blocks, Hkv), dtype=np.float32)
    vs = np.zeros((num_blocks, Hkv), dtype=np.float32)
    blk = (src_slots // BLOCK_SIZE).astype(np.int64)
    kabs = np.abs(bf16_to_f32(src_k)).max(axis=2)   # [N, Hkv]
    vabs = np.abs(bf16_to_f32(src_v)).max(axis=2)
    np.maximum.at(ks, blk, kabs)
    np.maximum.at(vs, blk, vabs)
    ks = np.where(ks > 0, ks / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    vs = np.where(vs > 0, vs / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    return ks, vs


def make_workload(name: str, *, context_lens, q_lens, num_q_heads: int, num_kv_heads: int,
                  head_dim: int, kv_dtype: str = "bf16", seed: int = 0, num_blocks: int | None = None,
                  pool_factor: float = 1.25, shared_prefix: list | None = None,
                  outlier_p: float = 0.0, scale: float | None = None) -> Workload:
    """Build a workload from explicit lengths.

    ``shared_prefix``: optional list of (first_seq, n_seqs, prefix_tokens) groups;
    the sequences of a group share the physical blocks of their first
    ``prefix_tokens`` tokens (a multiple of the block size), written once.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    L = np.asarray(context_lens, dtype=np.int32)
    Q = np.asarray(q_lens, dtype=np.int32)
    B = int(L.shape[0])
    Hkv, D = num_kv_heads, head_dim
    assert np.all(Q >= 0) and np.all(Q <= np.maximum(L, 0))
    nblk = (L.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE

    owner_prefix = np.zeros(B, dtype=np.int64)   # tokens of the prefix owned by another seq
    share_src = np.full(B, -1, dtype=np.int64)
    if shared_prefix:
        for first, n, ptoks in shared_prefix:
            assert ptoks % BLOCK_SIZE == 0
            for s in range(first + 1, first + n):
                owner_prefix[s] = ptoks
                share_src[s] = first
    private_blocks = nblk - owner_prefix // BLOCK_SIZE
    needed = int(private_blocks.sum())
    if num_blocks is None:
        num_blocks = max(int(np.ceil(needed * pool_factor)), needed, 1)
    assert num_blocks >= needed
    perm = rng.permutation(num_blocks).astype(np.int32)

    MB = max(int(nblk.max()) if B else 1, 1)
    tables = np.full((B, MB), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        shared = int(owner_prefix[b] // BLOCK_SIZE)
        if shared:
            tables[b, :shared] = tables[share_src[b], :shared]
        n_priv = int(nblk[b]) - shared
        tables[b, shared:nblk[b]] = perm[cursor:cursor + n_priv]
        cursor += n_priv

    # Tokens each sequence writes: positions [owner_prefix, L); the last Q of them
    # are the step's new tokens, the rest are prefill.
    pre_slots, step_slots = [], []
    for b in range(B):
        pos = np.arange(owner_prefix[b], L[b], dtype=np.int64)
        slots = tables[b, pos // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + pos % BLOCK_SIZE
        n_step = int(Q[b])
        pre_slots.append(slots[:len(slots) - n_step])
        step_slots.append(slots[len(slots) - n_step:])
    pre_slots = np.concatenate(pre_slots) if B else np.zeros(0, np.int64)
    step_slots = np.concatenate(step_slots) if B else np.zeros(0, np.int64)
    Np, T = int(pre_slots.shape[0]), int(step_slots.shape[0])

    # Draw in chunks to bound host memory at large sizes.
    def draw(n):
        out_k = np.empty((n, Hkv, D), dtype=np.uint16)
        out_v = np.empty((n, Hkv, D), dtype=np.uint16)
        chunk = max(1, (1 << 22) // max(1, Hkv * D))
        for s in range(0, n, chunk):
            e = min(n, s + chunk)
            out_k[s:e] = _normal_bf16(rng, (e - s, Hkv, D), outlier_p)
            out_v[s:e] = _normal_bf16(rng, (e - s, Hkv, D), outlier_p)
        return out_k, out_v

    pk, pv = draw(Np)
    q = _normal_bf16(rng, (T, num_q_heads, D))
    nk, nv = draw(T)

    ks = vs = None
    if kv_dtype == "fp8":
        ks, vs = _fp8_scales(num_blocks, Hkv, D, np.concatenate([pk, nk]), np.concatenate([pv, nv]),
                             np.concatenate([pre_slots, step_slots]))
    if scale is None:
        scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    return Workload(name=name, num_seqs=B, num_q_heads=num_q_heads, num_kv_heads=Hkv, head_dim=D,
                    kv_dtype=kv_dtype, scale=float(np.float32(scale)), num_blocks=num_blocks,
                    context_lens=L, q_lens=Q, block_tables=tables, prefill_k=pk, prefill_v=pv,
                    prefill_slots=pre_slots, q=q, k_new=nk, v_new=nv, slots=step_slots,
                    k_scales=ks, v_scales=vs, info={"seed": seed, "shared_prefix": list(shared_prefix or [])})


# ----------------------------------------------------------------------------------
# The five named configurations (seed = config number).
# ----------------------------------------------------------------------------------

def tiny_decode(seed: int = 1) -> Workload:
    """4 seqs, 8/2 heads, d=64, lens U[1,256], pool of 96 permuted blocks, q_len 1."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    L = rng.integers(1, 257, size=4).astype(np.int32)
    return make_workload("tiny_decode_b4_d64", context_lens=L, q_lens=np.ones(4, np.int32),
                         num_q_heads=8, num_kv_heads=2, head_dim=64, seed=seed, num_blocks=96)


def decode_b32_d128(seed: int = 2) -> Workload:
    """32 seqs, 32/8 heads, d=128, lens U[256,2048], 5,000-block shuffled pool."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    L = rng.integers(256, 2049, size=32).astype(np.int32)
    return make_workload("decode_b32_h32x8_d128", context_lens=L, q_lens=np.ones(32, np.int32),
                         num_q_heads=32, num_kv_heads=8, head_dim=128, seed=seed, num_blocks=5000)


def prefix_reuse_b32_d64(seed: int = 3) -> Workload:
    """8 conversations x 4 turns; shared prefix 512-1536 tokens (block aligned),
    private suffix U[32,256]; 32/8 heads, d=64."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    lens, groups = [], []
    for c in range(8):
        p = 16 * int(rng.integers(32, 97))
        groups.append((4 * c, 4, p))
        for _t in range(4):
            lens.append(p + int(rng.integers(32, 257)))
    L = np.asarray(lens, np.int32)
    return make_workload("prefix_reuse_8x4_d64", context_lens=L, q_lens=np.ones(32, np.int32),
                         num_q_heads=32, num_kv_heads=8, head_dim=64, seed=seed,
                         shared_prefix=groups, pool_factor=1.25)


def verify_b32_q5_d128(seed: int = 4) -> Workload:
    """32 seqs, 5-token causal verify window, lens U[512,4096], d=128."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    L = rng.integers(512, 4097, size=32).astype(np.int32)
    needed = int(((L + 15) // 16).sum())
    return make_workload("verify_b32_q5_d128", context_lens=L, q_lens=np.full(32, 5, np.int32),
                         num_q_heads=32, num_kv_heads=8, head_dim=128, seed=seed,
                         num_blocks=max(int(np.ceil(needed * 1.25)), 5000))


def long_fp8_b128_d128(seed: int = 5, num_seqs: int = 128, n_long: int = 4,
                       long_len: int = 32768) -> Workload:
    """128 seqs, log-normal lens (median 1024, sigma 1, clipped [16, 32768]),
    4 forced to 32768; FP8-e4m3 cache with per-(block, kv-head) scales."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    L = np.rint(np.exp(rng.normal(np.log(1024.0), 1.0, size=num_seqs)))
    L = np.clip(L, 16, 32768).astype(np.int32)
    idx = rng.choice(num_seqs, size=n_long, replace=False)
    L[idx] = long_len
    return make_workload("long_fp8_b128_d128", context_lens=L, q_lens=np.ones(num_seqs, np.int32),
                         num_q_heads=32, num_kv_heads=8, head_dim=128, kv_dtype="fp8", seed=seed,
                         pool_factor=1.1, outlier_p=0.01)


def long_prefix_reuse(prefix_tokens: int = 8192, seed: int = 7, conversations: int = 8,
                      turns: int = 4) -> Workload:
    """Conversations x turns sharing a long system prompt (prefix_tokens,
    block aligned) plus private suffixes U[32, 256]; 32/8 heads, d=64: the
    regime of the shared-prefix cascade (not one of the five named
    configurations)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens, groups = [], []
    for c in range(conversations):
        groups.append((turns * c, turns, prefix_tokens))
        for _ in range(turns):
            lens.append(prefix_tokens + int(rng.integers(32, 257)))
    return make_workload(f"long_prefix_{prefix_tokens}_{conversations}x{turns}_d64", context_lens=lens,
                         q_lens=[1] * len(lens), num_q_heads=32, num_kv_heads=8, head_dim=64, seed=seed,
                         shared_prefix=groups)


# The five named workloads, by number.
def prefill_b4_q2048_d128(seed: int = 8) -> Workload:
    """Four whole prompts of 2048 tokens processed at once (causal prefill):
    32 query / 8 KV heads, head_dim 128, bf16 K/V ~ N(0, 1), pages from a
    shuffled pool."""
    return make_workload("prefill_b4_q2048_d128", context_lens=[2048] * 4, q_lens=[2048] * 4,
                         num_q_heads=32, num_kv_heads=8, head_dim=128, seed=seed)


def chunked_prefill_b8_q512_d128(seed: int = 9) -> Workload:
    """Chunked prefill: eight sequences each appending a 512-token chunk after
    3584 resident tokens (context 4096); 32/8 heads, head_dim 128."""
    return make_workload("chunked_prefill_b8_q512_d128", context_lens=[4096] * 8, q_lens=[512] * 8,
                         num_q_heads=32, num_kv_heads=8, head_dim=128, seed=seed)


PREFILL_WORKLOADS = {
    "prefill_b4_q2048_d128": prefill_b4_q2048_d128,
    "chunked_prefill_b8_q512_d128": chunked_prefill_b8_q512_d128,
}


def causal_flops(w: Workload) -> int:
    """Multiply-add FLOPs of the attention's two products (q.k and p.v) over
    the keys each query sees: 4 * D * Hq per (query, visible key)."""
    L = w.context_lens.astype(np.int64)
    Q = w.q_lens.astype(np.int64)
    keys = Q * (L - Q) + Q * (Q + 1) // 2
    return int(4 * w.head_dim * w.num_q_heads * keys.sum())


WORKLOADS = {
    1: tiny_decode,
    2: decode_b32_d128,
    3: prefix_reuse_b32_d64,
    4: verify_b32_q5_d128,
    5: long_fp8_b128_d128,
}

"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

append: bit-exact whole cache buffers (bf16 and FP8), NaN sentinels included.
attention: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| element-wise, on the five
named configurations at full size (in the default launch configuration the
benchmark times) and on a sweep of small ragged shapes; plus invariants that
must hold bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import _native as nat
from paged_kv_decode_14_gb300 import workloads as wl
from paged_kv_decode_14_gb300.runner import DeviceWorkload
from gpu_helpers import (assert_attention_close, caches_equal, config_oracle, config_workload, out_bits,
                         to_f64)

pytestmark = pytest.mark.gpu


def run_gpu(w, num_ctas=0):
    dw = DeviceWorkload(w, num_ctas=num_ctas)
    dw.prefill()
    out = dw.step()
    torch.cuda.synchronize()
    return dw, out_bits(out)


# ------------------------------------------------------------------ named configs

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_config_append_and_attention(n):
    w = config_workload(n)
    kc, vc, ref, _ = config_oracle(n)
    dw, got = run_gpu(w)
    gk, gv = dw.cache_bytes()
    fp8 = w.kv_dtype == "fp8"
    assert caches_equal(gk, kc, fp8), "K cache differs from the oracle's"
    assert caches_equal(gv, vc, fp8), "V cache differs from the oracle's"
    assert_attention_close(got, ref, f"config {n}")
    assert dw.errors() == (0, 0)


def test_length_one_context_is_v_bitwise():
    w = wl.make_workload("l1", context_lens=[1, 1, 1], q_lens=[1, 1, 1], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, seed=61)
    _, got = run_gpu(w)
    G = 4
    for b in range(3):
        for h in range(8):
            assert np.array_equal(got[b, h], w.v_new[b, h // G])


# ------------------------------------------------------------------ small ragged sweep

SWEEP = [
    # (D, Hq, Hkv, lens, q_lens, dtype)
    (64, 8, 2, [1, 15, 16, 17, 31, 32, 33, 100], [1] * 8, "bf16"),
    (128, 8, 8, [1, 15, 16, 17, 64, 257], [1] * 6, "bf16"),
    (128, 8, 2, [5, 40, 77, 300], [5, 3, 8, 2], "bf16"),
    (128, 16, 2, [5, 40, 77, 300], [5, 3, 8, 2], "bf16"),  # G = 8, R up to 64: two virtual kv-heads per kv-head
    (64, 32, 2, [9, 130, 33], [4, 2, 3], "bf16"),          # G = 16, R up to 64
    (128, 32, 4, [20, 300], [5, 2], "fp8"),                # FP8, G = 8, Q = 5: four virtual groups of 10 rows
    (64, 4, 4, [9, 10, 11], [8, 4, 2], "bf16"),
    (128, 32, 8, [600, 3, 1200], [1, 1, 1], "fp8"),
    (64, 8, 1, [33, 17, 129], [4, 1, 2], "fp8"),           # FP8, G = 8, Q = 4: virtual groups of 2 heads
    (64, 8, 2, [50, 300, 700, 16], [9, 12, 16, 1], "fp8"),   # FP8, head_dim 64, 9-16 tokens: the CUDA-core kernel
    (128, 8, 2, [50, 300, 700, 16], [9, 12, 16, 1], "fp8"),  # FP8, head_dim 128, 16-token windows: 16-row segments
    (128, 32, 2, [1, 40, 333, 1030], [1, 1, 1, 1], "fp8"),   # FP8, G = 16: one 16-row segment per kv-head
    (128, 16, 1, [40, 250], [2, 2], "bf16"),          # G = 16, R = 32
    (128, 8, 2, [0, 20, 0, 45], [0, 1, 0, 2], "bf16"),  # empty sequences
    (64, 16, 2, [20, 50], [0, 3], "bf16"),             # a sequence with no query rows
    (128, 16, 2, [1, 15, 16, 17, 130, 700], [1] * 6, "fp8"),   # FP8, G = 8: one kv-head per segment
    (128, 8, 2, [5, 40, 77, 300], [2, 1, 2, 1], "fp8"),        # FP8, R = 8 with a causal window
    (128, 8, 4, [0, 33, 0, 517], [0, 1, 0, 1], "fp8"),         # FP8, empty sequences, four kv-heads per segment
    # FP8 with head_dim 64 on the tensor cores (1 KiB e4m3 pages, widened four pages a thread)
    (64, 32, 8, [1, 15, 16, 17, 130, 700, 2000], [1] * 7, "fp8"),   # G = 4: two kv-heads per segment
    (64, 16, 2, [5, 40, 77, 300], [1, 1, 1, 1], "fp8"),             # G = 8: one kv-head per segment
    (64, 8, 4, [9, 200, 33, 517], [2, 1, 4, 1], "fp8"),             # G = 2, causal windows, R <= 8
    (64, 8, 8, [0, 33, 0, 517, 64], [0, 1, 0, 1, 1], "fp8"),        # G = 1: four kv-heads per segment
    (64, 32, 8, np.random.default_rng(904).integers(1, 1500, 96).tolist(), [1] * 96, "fp8"),
    # wide segments of at most 24 columns (the 24-column softmax of the wide kernel)
    (128, 16, 4, [30, 300, 77, 1000], [3, 1, 2, 3], "bf16"),      # G = 4, R = 12: two kv-heads per segment
    (128, 16, 2, [50, 400, 9, 2000], [3, 2, 1, 3], "bf16"),       # G = 8, R = 24
    (128, 10, 2, [7, 333, 64, 1500], [2, 1, 2, 2], "bf16"),       # G = 5, R = 10: 20 columns, two kv-heads
    # verify windows (R = 20, wide segments: the weighted cut) over short and long sequences
    (128, 32, 8, [20, 700, 33, 17, 400, 90, 16, 1000], [5] * 8, "bf16"),
    # large batches: past the shared-memory sequence table (256 bf16 / 128 FP8
    # sequences) and past one planning chunk (384 sequences)
    (128, 32, 8, np.random.default_rng(901).integers(1, 81, 600).tolist(), [1] * 600, "bf16"),
    (128, 32, 8, np.random.default_rng(902).integers(1, 121, 200).tolist(), [1] * 200, "fp8"),
    (128, 32, 8, np.random.default_rng(903).integers(5, 61, 450).tolist(), [5] * 450, "bf16"),
]


@pytest.mark.parametrize("case", range(len(SWEEP)))
def test_sweep(case):
    D, Hq, Hkv, lens, ql, dt = SWEEP[case]
    w = wl.make_workload(f"sweep{case}", context_lens=lens, q_lens=ql, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, kv_dtype=dt, seed=100 + case, outlier_p=0.01 if dt == "fp8" else 0.0)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    for ncta in (0, 1, 3, 64):
        dw, got = run_gpu(w, num_ctas=ncta)
        gk, gv = dw.cache_bytes()
        assert caches_equal(gk, kc, dt == "fp8") and caches_equal(gv, vc, dt == "fp8")
        assert_attention_close(got, ref, f"sweep {case} ncta {ncta}")


def test_fp8_verify_q5_full_size():
    """FP8 cache, 5-token verify windows on the verify batch's shape (32
    sequences, lengths U[512, 4096], G = 4): R = 20 rows per kv-head run as
    two virtual groups of 10 on the wide FP8 tensor-core kernel."""
    rng = np.random.Generator(np.random.PCG64(1005))
    L = rng.integers(512, 4097, size=32).astype(np.int32)
    w = wl.make_workload("verify_fp8", context_lens=L, q_lens=np.full(32, 5, np.int32), num_q_heads=32,
                         num_kv_heads=8, head_dim=128, kv_dtype="fp8", seed=105, outlier_p=0.01)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_gpu(w)
    assert_attention_close(got, ref, "FP8 verify Q=5")
    assert dw.errors() == (0, 0)


def test_verify_g8_q5_full_size():
    """A 64 / 8-head model verifying 5 draft tokens on the verify batch's shape
    (32 sequences, lengths U[512, 4096]): R = G * Q = 40 rows per kv-head, so
    each kv-head's 8 query heads run as two virtual groups of 4."""
    rng = np.random.Generator(np.random.PCG64(1004))
    L = rng.integers(512, 4097, size=32).astype(np.int32)
    w = wl.make_workload("verify_g8", context_lens=L, q_lens=np.full(32, 5, np.int32), num_q_heads=64,
                         num_kv_heads=8, head_dim=128, seed=104)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_gpu(w)
    assert_attention_close(got, ref, "verify G=8 Q=5")
    assert dw.errors() == (0, 0)


def test_fp8_subnormal_codes():
    """Page scales 2^14 times absmax / 448 leave most stored codes e4m3
    subnormals (exponent field 0): the attention must decode them exactly."""
    w = wl.make_workload("fp8sub", context_lens=[300, 77, 1000, 16], q_lens=[1] * 4, num_q_heads=32,
                         num_kv_heads=8, head_dim=128, kv_dtype="fp8", seed=91)
    w.k_scales = (w.k_scales * np.float32(16384.0)).astype(np.float32)
    w.v_scales = (w.v_scales * np.float32(16384.0)).astype(np.float32)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_gpu(w)
    gk, gv = dw.cache_bytes()
    assert caches_equal(gk, kc, True) and caches_equal(gv, vc, True)
    written = np.concatenate([c[(c & 0x7F) != 0x7F] for c in (gk, gv)])   # (unwritten slots hold NaN)
    sub = (((written >> 3) & 15) == 0) & ((written & 7) != 0)
    assert np.mean(sub) > 0.3, "the case should hold mostly subnormal codes"
    assert_attention_close(got, ref, "fp8 subnormal codes")


@pytest.mark.parametrize("head_dim,group,num_kv_heads,dtype", [
    (128, 4, 2, "fp8"),     # tensor-core FP8 kernel, two kv-heads per segment
    (64, 4, 2, "fp8"),      # tensor-core FP8 kernel, head_dim 64
    (64, 16, 2, "fp8"),     # FP8, head_dim 64, G = 16: two virtual groups
    (128, 16, 2, "fp8"),    # FP8, G = 16: 16-row segments (the wide FP8 kernel)
    (128, 4, 2, "bf16"),    # tensor-core narrow kernel, two kv-heads per segment
    (64, 1, 4, "bf16"),     # narrow kernel, four kv-heads per segment
    (128, 16, 2, "bf16"),   # wide kernel (N = 32), two kv-heads per segment
    (128, 12, 2, "bf16"),   # wide kernel, 24 of its 32 columns (R = 12, two kv-heads per segment)
])
def test_nan_in_cache_propagates(head_dim, group, num_kv_heads, dtype):
    """A NaN source value is stored as NaN (bf16 bits copied; an E4M3 NaN code
    for FP8: the append keeps NaN).  Attention over it gives NaN exactly where
    the fp64 oracle does: every element of the rows whose K holds a NaN at a
    visible position, and the one dimension of the rows whose V does; the
    other kv-heads that share a segment, a tile and a P.V MMA with the NaN
    page stay finite."""
    Hkv = num_kv_heads
    w = wl.make_workload("nan", context_lens=[300, 77, 1000, 40], q_lens=[1, 1, 1, 1],
                         num_q_heads=Hkv * group, num_kv_heads=Hkv, head_dim=head_dim, kv_dtype=dtype,
                         seed=93, outlier_p=0.01 if dtype == "fp8" else 0.0)
    nan = np.uint16(0x7FC0)
    firsts = np.concatenate([[0], np.cumsum(w.context_lens - w.q_lens)])
    w.prefill_k = w.prefill_k.copy()
    w.prefill_v = w.prefill_v.copy()
    # K of sequence 0 at position 5 (kv-head 1), V of sequence 2 at position 600 (kv-head 0, dim 3)
    w.prefill_k[int(firsts[0]) + 5, 1, 7] = nan
    w.prefill_v[int(firsts[2]) + 600, 0, 3] = nan
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    assert np.isnan(ref).any() and not np.isnan(ref).all()
    dw, got = run_gpu(w)
    gk, gv = dw.cache_bytes()
    assert caches_equal(gk, kc, dtype == "fp8") and caches_equal(gv, vc, dtype == "fp8")
    assert_attention_close(got, ref, f"NaN {dtype} D={head_dim} G={group} Hkv={Hkv}", nan_aware=True)


@pytest.mark.parametrize("ncta", [1, 2, 3, 7, 152, 608, 5000])
def test_grid_sizes_agree(ncta):
    """Different grids cut the KV differently; the LSE merge makes them agree."""
    w = config_workload(2)
    _, _, ref, _ = config_oracle(2)
    _, base = run_gpu(w)
    _, got = run_gpu(w, num_ctas=ncta)
    a, b = to_f64(base), to_f64(got)
    # the splits only reorder fp32 sums: the bf16 outputs agree to two units in
    # the last place (2^-7 relative), plus a small absolute term for rows whose
    # value comes out of cancellation
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-4)
    assert_attention_close(got, ref, f"ncta {ncta}")


def test_identical_sequences_agree():
    """Sequences with the same block table, lengths and q rows give the same
    rows up to the order of the fp32 sums (they are cut at different points of
    the partition)."""
    w = wl.make_workload("twins", context_lens=[1000, 1000, 77, 1000, 333], q_lens=[1] * 5, num_q_heads=32,
                         num_kv_heads=8, head_dim=128, seed=61)
    for b in (1, 3):
        w.block_tables[b] = w.block_tables[0]
        w.q[b] = w.q[0]                               # (one q row per sequence)
    # the twins' new tokens land in sequence 0's slot, written once
    w.slots = w.slots.copy()
    w.slots[[1, 3]] = -1
    for ncta in (0, 7):
        _, got = run_gpu(w, num_ctas=ncta)
        g = to_f64(got)
        for b in (1, 3):
            assert np.all(np.abs(g[b] - g[0]) <= 2.0 ** -7 * np.maximum(np.abs(g[b]), np.abs(g[0])) + 1e-4)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    assert_attention_close(got, ref, "identical sequences")


# ------------------------------------------------------------------ invariants (bitwise)

def test_deterministic_run_to_run():
    w = config_workload(4)
    _, a = run_gpu(w)
    _, b = run_gpu(w)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_repeated_calls_reuse_the_workspace(n):
    """Calls that share a workspace give the same bits, and each call leaves
    every merge ticket at zero (the workspace is ready for the next call)."""
    w = config_workload(n)
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    first = out_bits(dw.attend())
    for _ in range(3):
        again = out_bits(dw.attend())
        assert np.array_equal(again, first)
    tickets = dw.workspace[256:256 + 4 * w.num_seqs * w.num_kv_heads].view(torch.int32)
    assert int(tickets.abs().sum().item()) == 0
    assert dw.errors() == (0, 0)


def test_block_permutation_invariance_bitwise():
    w = wl.make_workload("perm", context_lens=[70, 333, 128, 1000], q_lens=[1, 3, 2, 1], num_q_heads=16,
                         num_kv_heads=4, head_dim=128, seed=71, pool_factor=2.0)
    _, a = run_gpu(w)
    rng = np.random.default_rng(7)
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    w2 = wl.make_workload("perm", context_lens=[70, 333, 128, 1000], q_lens=[1, 3, 2, 1], num_q_heads=16,
                          num_kv_heads=4, head_dim=128, seed=71, pool_factor=2.0)
    w2.block_tables = np.where(w2.block_tables >= 0, perm[np.maximum(w2.block_tables, 0)], -1).astype(np.int32)
    w2.prefill_slots = perm[w2.prefill_slots // 16].astype(np.int64) * 16 + w2.prefill_slots % 16
    w2.slots = perm[w2.slots // 16].astype(np.int64) * 16 + w2.slots % 16
    _, b = run_gpu(w2)
    assert np.array_equal(a, b)


def test_shared_prefix_equals_private_copies_bitwise():
    lens = [16 * 40 + 50, 16 * 40 + 7, 16 * 40 + 200, 16 * 40 + 1]
    kw = dict(context_lens=lens, q_lens=[1] * 4, num_q_heads=32, num_kv_heads=8, head_dim=64, seed=72)
    shared = wl.make_workload("sh", shared_prefix=[(0, 4, 16 * 40)], **kw)
    private = wl.make_workload("pv", **kw)
    # same data: copy the shared prefix rows of sequence 0 into the private workload's other sequences
    _, a = run_gpu(shared)
    # build the private-copy version from the shared one: duplicate the prefix tokens per sequence
    nb_pref = 40
    w = shared
    tables = w.block_tables.copy()
    used = set(int(x) for x in tables[tables >= 0])
    free = [b for b in range(w.num_blocks + 200) if b not in used]
    extra_k, extra_v, extra_s = [], [], []
    pre_src = {}
    for t, s in enumerate(w.prefill_slots):
        pre_src[int(s)] = t
    for s in (1, 2, 3):
        for j in range(nb_pref):
            nb = free.pop(0)
            old = tables[s, j]
            tables[s, j] = nb
            for off in range(16):
                t = pre_src[int(old) * 16 + off]
                extra_k.append(w.prefill_k[t])
                extra_v.append(w.prefill_v[t])
                extra_s.append(nb * 16 + off)
    w.block_tables = tables
    w.num_blocks = w.num_blocks + 200
    w.prefill_k = np.concatenate([w.prefill_k, np.stack(extra_k)])
    w.prefill_v = np.concatenate([w.prefill_v, np.stack(extra_v)])
    w.prefill_slots = np.concatenate([w.prefill_slots, np.array(extra_s, np.int64)])
    _, b = run_gpu(w)
    assert np.array_equal(a, b)
    del private


def test_verify_row_equals_decode_call():
    """Verify row i == a decode call (Q=1) over the first L - Q + i + 1 tokens."""
    L, Q = 300, 5
    w = wl.make_workload("ver", context_lens=[L], q_lens=[Q], num_q_heads=8, num_kv_heads=2, head_dim=128,
                         seed=73)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    _, got = run_gpu(w)
    assert_attention_close(got, ref, "verify")
    for i in range(Q):
        wd = wl.make_workload("ver", context_lens=[L], q_lens=[Q], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=73)
        wd.context_lens = np.array([L - Q + i + 1], np.int32)
        wd.q_lens = np.array([1], np.int32)
        wd.q = w.q[i:i + 1].copy()
        keep = Q - i - 1        # the window tokens after i are not part of this context
        wd.k_new, wd.v_new, wd.slots = w.k_new[i:i + 1], w.v_new[i:i + 1], w.slots[i:i + 1]
        # prefill also holds the window tokens before i
        wd.prefill_k = np.concatenate([w.prefill_k, w.k_new[:i]])
        wd.prefill_v = np.concatenate([w.prefill_v, w.v_new[:i]])
        wd.prefill_slots = np.concatenate([w.prefill_slots, w.slots[:i]])
        del keep
        _, gd = run_gpu(wd)
        assert np.max(np.abs(to_f64(gd[0]) - to_f64(got[i]))) <= 2e-3 + 1e-2 * np.max(np.abs(to_f64(got[i])))


# ------------------------------------------------------------------ FP8 encode edges

@pytest.mark.parametrize("scale", [1.0, 0.5, 1.0 / 448.0, 3.7, 1e-3, 0.0826])
def test_fp8_append_every_bf16_pattern(scale):
    """All 65536 bf16 bit patterns (incl. inf, NaN, subnormals, -0) through the
    FP8 append, against the oracle encoder, at several scales (saturation
    at small scales)."""
    D, Hkv = 128, 1
    T = 65536 // D
    vals = np.arange(65536, dtype=np.uint16).reshape(T, Hkv, D)
    NB = (T + 15) // 16
    ks = np.full((NB, Hkv), scale, np.float32)
    kc = np.full(NB * Hkv * 16 * D, wl.FP8_NAN, np.uint8)
    vc = kc.copy()
    slots = np.arange(T, dtype=np.int64)
    oracle.paged_kv_append(1, kc, vc, ks, ks, NB, Hkv, D, vals, vals, slots)
    dev = "cuda"
    kst = torch.from_numpy(ks).to(dev)
    cache = nat.PagedKVCache(NB, Hkv, D, "fp8", device=dev, k_scales=kst, v_scales=kst)
    cache.k.fill_(0x7F)
    cache.v.fill_(0x7F)
    kt = torch.from_numpy(vals.view(np.int16)).to(dev).view(torch.bfloat16)
    nat.append(cache, kt, kt, torch.from_numpy(slots).to(dev))
    torch.cuda.synchronize()
    gk = cache.k.cpu().numpy().reshape(-1)
    assert caches_equal(gk, kc, True)


def test_append_skips_negative_slots_and_flags_out_of_range():
    D, Hkv, NB = 64, 2, 4
    w_k = np.arange(3 * Hkv * D, dtype=np.uint16).reshape(3, Hkv, D)
    dev = "cuda"
    cache = nat.PagedKVCache(NB, Hkv, D, "bf16", device=dev)
    cache.k.view(torch.int16).fill_(0x7FC0)
    cache.v.view(torch.int16).fill_(0x7FC0)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kt = torch.from_numpy(w_k.view(np.int16)).to(dev).view(torch.bfloat16)
    slots = torch.tensor([-1, NB * 16 + 3, 5], dtype=torch.int64, device=dev)
    nat.append(cache, kt, kt, slots, device_error=err)
    assert nat.read_device_error(err) == nat.DEVERR_SLOT
    kc = np.full(NB * Hkv * 16 * D, wl.BF16_NAN, np.uint16)
    vc = kc.copy()
    oracle.paged_kv_append(0, kc, vc, None, None, NB, Hkv, D, w_k, w_k, slots.cpu().numpy())
    got = cache.k.view(torch.int16).cpu().numpy().reshape(-1).view(np.uint16)
    assert np.array_equal(got, kc)


def test_fp8_v_scale_range():
    """FP8 caches take P.V in fp16 with P carrying the page's v scale: a
    scale of 255 (P < 2^8 keeps P * scale inside fp16) matches the oracle
    with no error; 256 sets PKV_DEVERR_RANGE."""
    w = wl.make_workload("f8range", context_lens=[300, 77], q_lens=[1, 1], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, kv_dtype="fp8", seed=950)
    blk = int(w.block_tables[0, 3])
    w.v_scales[blk, 2] = 255.0
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_gpu(w)
    assert_attention_close(got, ref, "v scale 255")
    assert dw.errors() == (0, 0)
    w.v_scales[blk, 2] = 256.0
    dw, _ = run_gpu(w)
    a, _ = dw.errors()
    assert a == nat.DEVERR_RANGE

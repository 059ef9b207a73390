"""GPU parity of the paged chunked-prefill kernel (pkv_paged_prefill) against
the CPU oracle's paged attention, which takes any query window: whole
prompts (Q = L), chunks appended after a resident context (Q < L), ragged
batches mixing windows of 1 .. 513 tokens with empty sequences, GQA groups
1 .. 16, head_dim 64 and 128, pages scattered through the pool.  Tolerance
as for the decode kernels: |gpu - oracle| <= 2e-3 + 1e-2 |oracle|."""

import copy

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import _native as nat
from paged_kv_decode_14_gb300 import workloads as wl
from paged_kv_decode_14_gb300.runner import DeviceWorkload
from gpu_helpers import assert_attention_close, out_bits

pytestmark = pytest.mark.gpu


def run_prefill(w):
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    out = dw.attend_prefill()
    torch.cuda.synchronize()
    return dw, out_bits(out)


CASES = [
    # (name, D, Hq, Hkv, context_lens, q_lens)
    ("prompt_g4_d128", 128, 8, 2, [300], [300]),                          # one whole prompt, ragged last tile
    ("chunk_g8_d128", 128, 32, 4, [956], [256]),                          # 256 new tokens after 700 resident
    ("ragged_g2_d64", 64, 8, 4, [1, 40, 0, 128, 600, 50], [1, 17, 0, 128, 513, 0]),
    ("prompt_g1_d64", 64, 4, 4, [200], [200]),                            # MHA: 128 positions per CTA
    ("prompt_g16_d128", 128, 32, 2, [333, 129], [333, 64]),               # 8 positions per CTA
    ("chunks_g4_d128", 128, 16, 4, [2100, 517, 16, 17], [129, 500, 16, 3]),
    ("page_edges_g8_d64", 64, 16, 2, [15, 16, 17, 127, 128, 129, 255], [15, 16, 17, 127, 128, 1, 200]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_matches_oracle(case):
    name, D, Hq, Hkv, L, Q = case
    w = wl.make_workload(name, context_lens=L, q_lens=Q, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                         seed=700 + CASES.index(case))
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_prefill(w)
    assert_attention_close(got, ref, name)
    assert dw.errors() == (0, 0)


def test_prefill_b4_2048_full_size():
    """Four 2048-token prompts of a 32 / 8-head, head_dim 128 model (the
    prefill benchmark's shape): 64 query blocks per (sequence, kv-head)."""
    w = wl.make_workload("prefill_b4", context_lens=[2048] * 4, q_lens=[2048] * 4, num_q_heads=32,
                         num_kv_heads=8, head_dim=128, seed=710)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_prefill(w)
    assert_attention_close(got, ref, "prefill B=4 Q=L=2048")
    assert dw.errors() == (0, 0)


def test_prefill_deterministic_and_placement_free():
    """Two calls give the same bits, and moving every page to another
    physical block (the pool permuted: tables and slots remapped together)
    changes nothing."""
    w = wl.make_workload("det", context_lens=[700, 300], q_lens=[400, 300], num_q_heads=16, num_kv_heads=4,
                         head_dim=128, seed=711)
    dw, a = run_prefill(w)
    b = out_bits(dw.attend_prefill())
    assert np.array_equal(a, b)
    perm = np.random.default_rng(5).permutation(w.num_blocks).astype(np.int32)
    w2 = copy.copy(w)
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    w2.prefill_slots = perm[w.prefill_slots // 16].astype(np.int64) * 16 + w.prefill_slots % 16
    w2.slots = perm[w.slots // 16].astype(np.int64) * 16 + w.slots % 16
    assert not np.array_equal(w2.block_tables, w.block_tables)
    _, c = run_prefill(w2)
    assert np.array_equal(a, c)


def test_prefill_agrees_with_verify_kernel_on_short_windows():
    """On windows the verify kernel also takes (Q <= 16) both kernels meet the
    oracle; a one-token window over one key returns that key's V row."""
    w = wl.make_workload("short", context_lens=[1, 90, 400], q_lens=[1, 16, 5], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, seed=712)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_prefill(w)
    assert_attention_close(got, ref, "prefill kernel, short windows")
    assert_attention_close(out_bits(dw.attend()), ref, "verify kernel, short windows")
    for h in range(8):
        assert np.array_equal(got[0, h], w.v_new[0, h // 4])


def test_prefill_rejections():
    w = wl.make_workload("rej", context_lens=[40], q_lens=[40], num_q_heads=8, num_kv_heads=2, head_dim=64,
                         seed=713)
    dw = DeviceWorkload(w)
    c = dw.cache
    # G = 3 does not divide 128
    q3 = torch.zeros(40, 6, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nat.PagedKVError) as e:
        nat.prefill(c, q3, dw.block_tables, dw.context_lens, dw.q_lens, 40, 0.1)
    assert e.value.status == 2
    # FP8 caches are not taken
    f8 = nat.PagedKVCache(w.num_blocks, 2, 64, "fp8", device="cuda",
                          k_scales=torch.ones(w.num_blocks, 2, device="cuda"),
                          v_scales=torch.ones(w.num_blocks, 2, device="cuda"))
    with pytest.raises(nat.PagedKVError) as e:
        nat.prefill(f8, dw.q, dw.block_tables, dw.context_lens, dw.q_lens, 40, 0.1)
    assert e.value.status == 2
    # no sequences: nothing launched, OK
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    nat.prefill(c, dw.q, dw.block_tables[:0], z, z, 1, 0.1)
    torch.cuda.synchronize()


def test_prefill_device_errors_are_reported_without_fault():
    """A block id outside the pool and a window longer than its context set
    the error word's bits; the kernel skips them (no fault) and later calls
    on the same context are exact."""
    w = wl.make_workload("errs", context_lens=[300, 200], q_lens=[300, 100], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, seed=714)
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    bt = dw.block_tables.clone()
    bt[0, 3] = w.num_blocks + 5
    nat.prefill(dw.cache, dw.q, bt, dw.context_lens, dw.q_lens, 300, w.scale, device_error=dw.prefill_err)
    assert nat.read_device_error(dw.prefill_err) == nat.DEVERR_BLOCK_ID
    ql = dw.q_lens.clone()
    ql[1] = 250                      # > context 200 (q rows still fit: 300 + 250 > 400 is not read past)
    ql[0] = 150
    nat.prefill(dw.cache, dw.q, dw.block_tables, dw.context_lens, ql, 300, w.scale, device_error=dw.prefill_err)
    assert nat.read_device_error(dw.prefill_err) == nat.DEVERR_LENGTH
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    assert_attention_close(out_bits(dw.attend_prefill()), ref, "after device errors")
    assert dw.errors() == (0, 0)


def test_prefill_wait_timeout_reports_and_recovers():
    """The bounded waits of the prefill kernel, made to run out without a
    fault: a 200 us limit and a hold flag that nothing sets.  The producer
    gives up, raises PKV_DEVERR_TIMEOUT, every role winds down, and the next
    call gives oracle parity."""
    w = wl.make_workload("to_pf", context_lens=[600, 300], q_lens=[600, 100], num_q_heads=16, num_kv_heads=4,
                         head_dim=128, seed=715)
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    hold = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        nat.debug_set_wait_limit(200_000, hold)
        dw.attend_prefill()
        torch.cuda.synchronize()
    finally:
        nat.debug_set_wait_limit(0, None)
    assert nat.read_device_error(dw.prefill_err) == nat.DEVERR_TIMEOUT
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    assert_attention_close(out_bits(dw.attend_prefill()), ref, "after a timeout")
    assert dw.errors() == (0, 0)


def test_prefill_large_logit_jumps():
    """A key whose logits jump by tens of octaves (K = +-40 in every
    dimension) far from the causal diagonal: rows whose running maximum
    rises by more than 2^32 inside a tile re-reference the P already written
    (exact power-of-two scaling), rows rising by 2^8 .. 2^32 rescale at the
    next tile, and all stay within the tolerance of the fp64 oracle."""
    w = wl.make_workload("jumps", context_lens=[1500, 900], q_lens=[300, 200], num_q_heads=16, num_kv_heads=4,
                         head_dim=128, seed=716)
    big, neg = np.uint16(0x4220), np.uint16(0xC220)        # bf16 40.0 and -40.0
    w.prefill_k[600] = big                                 # sequence 0, position 600 (key tile 4)
    w.prefill_k[1000] = neg                                # sequence 0, position 1000
    w.prefill_k[1200 + 350] = big                          # sequence 1, position 350 (its prefill starts at 1200)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_prefill(w)
    assert_attention_close(got, ref, "large logit jumps")
    assert dw.errors() == (0, 0)


def test_prefill_v_beyond_fp16_range_is_reported():
    """The P.V products run in fp16: a finite V value of magnitude >= 65536
    (here 98304) cannot be carried and sets PKV_DEVERR_RANGE; values just
    inside the range (65280, the largest bf16 below 65504) are exact."""
    w = wl.make_workload("range", context_lens=[300], q_lens=[100], num_q_heads=8, num_kv_heads=2, head_dim=64,
                         seed=717)
    w.prefill_v[50, 1, 7] = np.uint16(0x477F)              # 65280: inside the fp16 range
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw, got = run_prefill(w)
    assert_attention_close(got, ref, "V = 65280")
    assert dw.errors() == (0, 0)
    w.prefill_v[60, 0, 3] = np.uint16(0x47C0)              # 98304
    dw, _ = run_prefill(w)
    a, _ = dw.errors()
    assert a == nat.DEVERR_RANGE


def test_prefill_nan_in_k_reaches_exactly_the_rows_that_see_it():
    """A NaN stored in K makes every element of the rows that see that key
    NaN (as in the definition) and leaves every other row exact: keys in
    the one-pass tiles and on the causal diagonal, rows sharing a warp."""
    w = wl.make_workload("nan_k", context_lens=[700, 400], q_lens=[500, 400], num_q_heads=16, num_kv_heads=4,
                         head_dim=128, seed=718)
    w.prefill_k[100, 2, 5] = np.uint16(0x7FC0)            # sequence 0, position 100 (resident), kv-head 2
    w.k_new[300, 1, 0] = np.uint16(0x7FC0)                # sequence 0, position 500 (in the window), kv-head 1
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    assert np.isnan(ref).any() and not np.isnan(ref).all()
    dw, got = run_prefill(w)
    assert_attention_close(got, ref, "NaN in K", nan_aware=True)

"""Fused RoPE + append (pkv_paged_kv_append_rope) against the oracle: the
cache (rotated K, V, FP8 codes), the rotated q and the FP8 scales chosen from
the values bit for bit, and attention over the result within the attention
tolerance.  Prefill and step go through separate calls, as a serving loop
makes them (the step's tokens may start new blocks)."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import _native as nat
from paged_kv_decode_14_gb300 import workloads as wl
from paged_kv_decode_14_gb300.runner import DeviceWorkload, _bf16_tensor
from gpu_helpers import assert_attention_close, caches_equal, out_bits

pytestmark = pytest.mark.gpu


def _positions(w):
    """Position of every prefill token and every step token in its sequence."""
    pre, step = [], []
    for L, Q in zip(w.context_lens.tolist(), w.q_lens.tolist()):
        pre.append(np.arange(0, L - Q))
        step.append(np.arange(L - Q, L))
    return np.concatenate(pre).astype(np.int32), np.concatenate(step).astype(np.int32)


def _run(w, theta, rotate, autoscale, pos_offset=0):
    kd = oracle.KV_FP8 if w.kv_dtype == "fp8" else oracle.KV_BF16
    pos_pre, pos_step = _positions(w)
    pos_pre, pos_step = pos_pre + pos_offset, pos_step + pos_offset
    # oracle side
    kc, vc = w.empty_cache(), w.empty_cache()
    ks = None if w.k_scales is None else w.k_scales.copy()
    vs = None if w.v_scales is None else w.v_scales.copy()
    q_ref = oracle.rope(w.q, pos_step, theta) if rotate else w.q
    for k, v, slots, pos in ((w.prefill_k, w.prefill_v, w.prefill_slots, pos_pre), (w.k_new, w.v_new, w.slots, pos_step)):
        kr = oracle.rope(k, pos, theta) if rotate else k
        if autoscale:
            oracle.fp8_autoscale(kr, v, slots, w.num_blocks, ks, vs)
        oracle.paged_kv_append(kd, kc, vc, ks, vs, w.num_blocks, w.num_kv_heads, w.head_dim, kr, v, slots)
    ref, _ = oracle.paged_attention(kd, kc, vc, ks, vs, w.num_blocks, w.num_kv_heads, w.head_dim, q_ref, w.num_q_heads,
                                    w.block_tables, w.context_lens, w.q_lens, w.scale)
    # GPU side
    dw = DeviceWorkload(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = torch.device("cuda")
    nat.append_rope(dw.cache, _bf16_tensor(w.prefill_k, dev), _bf16_tensor(w.prefill_v, dev),
                    torch.from_numpy(w.prefill_slots).to(dev), torch.from_numpy(pos_pre).to(dev) if rotate else None,
                    theta, fp8_scales_from_values=autoscale, device_error=err)
    nat.append_rope(dw.cache, dw.k_new, dw.v_new, dw.slots, torch.from_numpy(pos_step).to(dev) if rotate else None,
                    theta, q=dw.q if rotate else None, fp8_scales_from_values=autoscale, device_error=err)
    out = dw.attend()
    torch.cuda.synchronize()
    gk, gv = dw.cache_bytes()
    fp8 = w.kv_dtype == "fp8"
    assert caches_equal(gk, kc, fp8), "K cache differs from the oracle's"
    assert caches_equal(gv, vc, fp8), "V cache differs from the oracle's"
    assert np.array_equal(dw.q.view(torch.int16).cpu().numpy().view(np.uint16), q_ref), "rotated q differs"
    if autoscale:
        assert np.array_equal(dw.cache.k_scales.cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(dw.cache.v_scales.cpu().numpy().view(np.uint32), vs.view(np.uint32))
    assert_attention_close(out_bits(out), ref, f"rope {w.kv_dtype} rotate={rotate} autoscale={autoscale}")
    assert nat.read_device_error(err) == 0
    assert dw.errors() == (0, 0)


def _workload(dtype, seed, D=128, lens=(300, 77, 1000, 40, 16, 17), ql=(1, 1, 2, 1, 1, 3)):
    return wl.make_workload("rope", context_lens=list(lens), q_lens=list(ql), num_q_heads=32, num_kv_heads=8,
                            head_dim=D, kv_dtype=dtype, seed=seed, outlier_p=0.01 if dtype == "fp8" else 0.0)


def test_rope_append_bf16():
    _run(_workload("bf16", 201), 10000.0, rotate=True, autoscale=False)


def test_rope_append_bf16_head_dim_64_large_positions():
    """Positions past 65 000 (angles in fp64), head_dim 64, theta 1e6."""
    _run(_workload("bf16", 202, D=64), 1.0e6, rotate=True, autoscale=False, pos_offset=65000)


def test_rope_append_fp8_scales_from_values():
    w = _workload("fp8", 203)
    w.k_scales[:] = 1.0                         # replaced for every block the calls start
    w.v_scales[:] = 1.0
    _run(w, 10000.0, rotate=True, autoscale=True)


def test_fp8_scales_from_values_without_rotation():
    w = _workload("fp8", 204, D=64)
    w.k_scales[:] = 3.0
    w.v_scales[:] = 3.0
    _run(w, 10000.0, rotate=False, autoscale=True)


def test_rope_append_fp8_given_scales():
    _run(_workload("fp8", 205), 10000.0, rotate=True, autoscale=False)


def test_rope_append_then_attention_large_batch():
    """300 sequences: the RoPE append (one CTA per token) runs long enough
    that an attention launched before it ended would read q rows not yet
    rotated; the attention must see every rotated row."""
    rng = np.random.default_rng(206)
    lens = rng.integers(4, 400, 300).tolist()
    ql = [int(min(L, 1 + (i % 3))) for i, L in enumerate(lens)]
    _run(_workload("bf16", 206, lens=lens, ql=ql), 10000.0, rotate=True, autoscale=False)

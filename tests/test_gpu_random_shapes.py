"""Seeded random shapes against the oracle.  Decode / verify: head_dim 64 or
128, GQA groups 1-16, windows of 1-16 tokens, bf16 and FP8 caches, ragged
lengths (empty and one-token sequences included), two grid sizes; every
kernel instance the planner can pick (narrow and wide bf16, the 20-column
wide instance, FP8 8- and 16-row segments, virtual groups, the CUDA-core FP8
kernel) is reached by some case.  Prefill: whole prompts and chunks after a
resident context, GQA groups 1-32, head_dim 64 and 128."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import workloads as wl
from paged_kv_decode_14_gb300.runner import DeviceWorkload
from gpu_helpers import assert_attention_close, caches_equal, out_bits

pytestmark = pytest.mark.gpu


def run_gpu(w, num_ctas=0):
    dw = DeviceWorkload(w, num_ctas=num_ctas)
    dw.prefill()
    out = dw.step()
    torch.cuda.synchronize()
    return dw, out_bits(out)

GROUPS = [1, 2, 3, 4, 5, 6, 8, 10, 12, 16]


def _case(i):
    rng = np.random.default_rng(5000 + i)
    D = int(rng.choice([64, 128]))
    dt = "fp8" if rng.random() < 0.5 else "bf16"
    G = int(rng.choice(GROUPS))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 9))
    qmax = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 9, 12, 16]))
    lens, ql = [], []
    for _ in range(B):
        L = int(rng.choice([0, 1, int(rng.integers(2, 40)), int(rng.integers(40, 700))]))
        Q = 0 if L == 0 else int(rng.integers(1, min(qmax, L) + 1))
        lens.append(L)
        ql.append(Q)
    if max(ql) == 0:
        lens[0], ql[0] = max(lens[0], 5), 1
    return D, dt, G * Hkv, Hkv, lens, ql


@pytest.mark.parametrize("i", range(40))
def test_random_shape(i):
    D, dt, Hq, Hkv, lens, ql = _case(i)
    w = wl.make_workload(f"rand{i}", context_lens=lens, q_lens=ql, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, kv_dtype=dt, seed=6000 + i, outlier_p=0.01 if dt == "fp8" else 0.0)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    for ncta in (0, 5):
        dw, got = run_gpu(w, num_ctas=ncta)
        gk, gv = dw.cache_bytes()
        assert caches_equal(gk, kc, dt == "fp8") and caches_equal(gv, vc, dt == "fp8")
        assert_attention_close(got, ref, f"random {i}: D={D} {dt} Hq={Hq} Hkv={Hkv} Q={ql} ncta={ncta}")
        assert dw.errors() == (0, 0)


def _prefill_case(i):
    rng = np.random.default_rng(7000 + i)
    D = int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 4, 8, 16, 32]))
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 5))
    lens, ql = [], []
    for _ in range(B):
        L = int(rng.choice([0, int(rng.integers(1, 64)), int(rng.integers(64, 900))]))
        Q = 0 if L == 0 else int(rng.choice([L, int(rng.integers(1, L + 1))]))
        lens.append(L)
        ql.append(Q)
    if max(ql) == 0:
        lens[0], ql[0] = 100, 100
    return D, G * Hkv, Hkv, lens, ql


@pytest.mark.parametrize("i", range(24))
def test_random_prefill_shape(i):
    """pkv_paged_prefill on random windows (whole prompts and chunks after a
    resident context, 1 to ~900 tokens), GQA groups 1-32, head_dim 64/128."""
    D, Hq, Hkv, lens, ql = _prefill_case(i)
    w = wl.make_workload(f"randpf{i}", context_lens=lens, q_lens=ql, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, seed=8000 + i)
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    got = out_bits(dw.attend_prefill())
    torch.cuda.synchronize()
    assert_attention_close(got, ref, f"random prefill {i}: D={D} Hq={Hq} Hkv={Hkv} L={lens} Q={ql}")
    assert dw.errors() == (0, 0)

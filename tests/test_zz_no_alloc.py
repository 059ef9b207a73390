"""pkv_paged_attention_noalloc: the attention entry point for callers that
cannot allocate device memory (a host that can only pass the tensors it
already holds, or a serving loop with a device budget fixed at start-up).  It
keeps its scratch in the library's static device array instead of a
caller-provided workspace.

Checked through the C ABI against pkv_paged_attention (the entry point with a
caller workspace), bit for bit, on two calls in a row (the second call reuses
the array the first one left behind), and against the oracle within the
attention tolerance; bf16 and FP8 caches on both kernels.  The
file sorts last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import _native as nat
from paged_kv_decode_14_gb300 import workloads as wl
from paged_kv_decode_14_gb300.runner import DeviceWorkload

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def _f64(t):
    return wl.bf16_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def _case(which):
    if which == "decode":
        return wl.decode_b32_d128()
    if which == "verify":
        return wl.make_workload("v", context_lens=[700, 45, 2100, 16], q_lens=[5, 5, 3, 1], num_q_heads=32,
                                num_kv_heads=8, head_dim=128, seed=91)
    if which == "fp8_tc":        # FP8, head_dim 128, G * Q <= 8: the tensor-core kernel
        return wl.make_workload("f8", context_lens=[900, 33, 1700, 5], q_lens=[1, 1, 1, 1], num_q_heads=32,
                                num_kv_heads=8, head_dim=128, kv_dtype="fp8", seed=92, outlier_p=0.01)
    if which == "fp8_tc64":      # FP8, head_dim 64, G * Q = 8: the tensor-core kernel
        return wl.make_workload("f8t", context_lens=[900, 33, 1700, 5], q_lens=[1, 2, 1, 1], num_q_heads=32,
                                num_kv_heads=8, head_dim=64, kv_dtype="fp8", seed=94, outlier_p=0.01)
    # FP8, head_dim 64, a 9-token window: the CUDA-core kernel (its own rows_pad and grid of 4 CTAs per SM)
    return wl.make_workload("f8s", context_lens=[900, 33, 1700, 9], q_lens=[1, 9, 1, 1], num_q_heads=32,
                            num_kv_heads=8, head_dim=64, kv_dtype="fp8", seed=93, outlier_p=0.01)


@pytest.mark.parametrize("which", ["decode", "verify", "fp8_tc", "fp8_tc64", "fp8_simt"])
def test_noalloc_matches_workspace_entry_two_calls(which):
    """Two calls in a row, each bit-identical to pkv_paged_attention with a
    caller workspace (the same kernel, grid and partition, so the same sums
    in the same order); the first also within the tolerance of the oracle."""
    w = _case(which)
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    ref = dw.attend().clone()
    torch.cuda.synchronize()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(dw.q, float("nan"))
        nat.attention_noalloc(dw.cache, dw.q, dw.block_tables, dw.context_lens, dw.q_lens, max(1, w.max_q_len),
                              w.scale, out=out, device_error=err)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}: differs from the workspace entry"
        assert nat.read_device_error(err) == 0
        if call == 0:
            kc, vc = oracle.build_cache(w)
            exp, _ = oracle.attend(w, kc, vc)
            a = _f64(out)
            assert np.all(np.abs(a - exp) <= ATOL + RTOL * np.abs(exp)), f"max err vs oracle {np.abs(a - exp).max()}"


def test_noalloc_rejects_sizes_beyond_its_array():
    w = wl.tiny_decode()
    dw = DeviceWorkload(w)
    with pytest.raises(nat.PagedKVError) as e:
        # a grid this large needs far more partial slots than the static array holds
        nat.attention_noalloc(dw.cache, dw.q, dw.block_tables, dw.context_lens, dw.q_lens, 1, w.scale,
                              num_ctas=1 << 20)
    assert e.value.status == 3

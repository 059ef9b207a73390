"""Shared-prefix cascade (pkv_paged_attention_cascade): the prefix of each
group of sequences attended once for the whole group, then each sequence's
own pages, merged per row.  Against the oracle on the prefix-reuse workload
at full size and on ragged groups (no prefix, single-sequence groups, verify
windows, head_dim 64 and 128), and against the plain attention over the same
tables."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import _native as nat
from paged_kv_decode_14_gb300 import workloads as wl
from paged_kv_decode_14_gb300.runner import DeviceWorkload
from gpu_helpers import assert_attention_close, config_oracle, config_workload, out_bits, to_f64

pytestmark = pytest.mark.gpu


def _check(w, ref=None):
    if ref is None:
        kc, vc = oracle.build_cache(w)
        ref, _ = oracle.attend(w, kc, vc)
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    plain = out_bits(dw.attend()).copy()
    got = out_bits(dw.attend_cascade(out=torch.empty_like(dw.q)))
    torch.cuda.synchronize()
    assert_attention_close(got, ref, f"cascade {w.name}")
    # the same attention as the plain call, summed in another order
    a, b = to_f64(got), to_f64(plain)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-4)
    assert nat.read_device_error(dw.cascade_ws) == 0
    return dw, got


def test_cascade_prefix_reuse_full_size():
    _, _, ref, _ = config_oracle(3)
    _check(config_workload(3), ref)


@pytest.mark.parametrize("D", [64, 128])
def test_cascade_ragged_groups(D):
    # groups: 3 turns sharing 5 blocks, a sequence alone, 2 turns sharing 1 block,
    # a one-sequence "group" with a 2-block prefix, 2 turns sharing 0 blocks
    lens = [80 + 7, 80 + 40, 80 + 1, 50, 16 + 9, 16 + 300, 32 + 3, 20, 33]
    ql = [1, 1, 1, 1, 1, 1, 1, 1, 1]
    groups = [(0, 3, 80), (4, 2, 16), (6, 1, 32)]
    w = wl.make_workload(f"casc{D}", context_lens=lens, q_lens=ql, num_q_heads=16, num_kv_heads=4, head_dim=D,
                         seed=301 + D, shared_prefix=groups)
    _check(w)


def test_cascade_verify_windows():
    """Turns verifying 5 draft tokens after a shared prefix (the window lies
    after the prefix)."""
    lens = [16 * 30 + 9, 16 * 30 + 60, 16 * 30 + 5, 200, 16 * 8 + 100]
    ql = [5, 5, 5, 5, 3]
    w = wl.make_workload("cascv", context_lens=lens, q_lens=ql, num_q_heads=8, num_kv_heads=2, head_dim=128,
                         seed=311, shared_prefix=[(0, 3, 16 * 30)])
    _check(w)


def test_cascade_rejects_a_partial_block_prefix():
    w = wl.make_workload("cascbad", context_lens=[100, 120], q_lens=[1, 1], num_q_heads=8, num_kv_heads=2,
                         head_dim=64, seed=321, shared_prefix=[(0, 2, 64)])
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    dw.attend_cascade()
    dw.group_prefix_lens[0] = 60                # not a multiple of 16
    dw.attend_cascade()
    torch.cuda.synchronize()
    assert nat.read_device_error(dw.cascade_ws) & nat.DEVERR_LENGTH

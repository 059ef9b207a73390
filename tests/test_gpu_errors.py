"""Error behaviour of the C ABI on the GPU: host-side argument checks return
a status and launch nothing; device-side bad indices set the error word and
never fault; the workspace stays usable afterwards."""

import numpy as np
import pytest
import torch

from paged_kv_decode_14_gb300 import _native as nat
from paged_kv_decode_14_gb300 import workloads as wl
from paged_kv_decode_14_gb300.runner import DeviceWorkload
from gpu_helpers import assert_attention_close, out_bits
import oracle

pytestmark = pytest.mark.gpu


def small():
    return wl.make_workload("e", context_lens=[40, 90], q_lens=[1, 2], num_q_heads=8, num_kv_heads=2,
                            head_dim=64, seed=81)


def test_host_checks_return_status():
    dw = DeviceWorkload(small())
    dw.prefill()
    c = dw.cache
    with pytest.raises(nat.PagedKVError) as e:      # workspace too small
        nat.attention(c, dw.q, dw.block_tables, dw.context_lens, dw.q_lens, 2, 0.1, dw.workspace[:64])
    assert e.value.status == 3
    with pytest.raises(nat.PagedKVError) as e:      # Hq not a multiple of Hkv
        nat.attention(c, dw.q[:, :7].contiguous(), dw.block_tables, dw.context_lens, dw.q_lens, 2, 0.1,
                      dw.workspace)
    assert e.value.status == 1
    bad = nat.PagedKVCache(c.num_blocks, c.num_kv_heads, 96, "bf16")    # head_dim 96 not built
    with pytest.raises(nat.PagedKVError) as e:
        nat.attention(bad, dw.q, dw.block_tables, dw.context_lens, dw.q_lens, 2, 0.1, dw.workspace)
    assert e.value.status == 2
    with pytest.raises(nat.PagedKVError) as e:      # max_q_len above the supported window
        nat.attention(c, dw.q, dw.block_tables, dw.context_lens, dw.q_lens, 17, 0.1, dw.workspace)
    assert e.value.status == 2
    wide = torch.full((2, (1 << 20) // c.num_kv_heads), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(nat.PagedKVError) as e:      # max_blocks_per_seq * Hkv beyond 2^20 units per sequence
        nat.attention(c, dw.q, wide, dw.context_lens, dw.q_lens, 2, 0.1, dw.workspace)
    assert e.value.status == 2


def test_bad_block_id_sets_error_word_then_recovers():
    w = small()
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    good = dw.block_tables.clone()
    dw.block_tables[1, 2] = w.num_blocks + 7
    dw.attend()
    torch.cuda.synchronize()
    attn_err, _ = dw.errors()
    assert attn_err & nat.DEVERR_BLOCK_ID
    dw.block_tables.copy_(good)
    dw.block_tables[0, 0] = -3
    dw.attend()
    assert dw.errors()[0] & nat.DEVERR_BLOCK_ID
    # the same workspace gives correct results once the table is fixed
    dw.block_tables.copy_(good)
    out = dw.attend()
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    assert_attention_close(out_bits(out), ref, "after recovery")
    assert dw.errors() == (0, 0)


def test_q_len_above_context_len_sets_error_word():
    w = small()
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    dw.context_lens[1] = 1     # q_lens[1] = 2 > context_lens[1]; q stays packed as before
    dw.attend()
    assert dw.errors()[0] & nat.DEVERR_LENGTH


def test_empty_batch_is_noop():
    w = small()
    dw = DeviceWorkload(w)
    c = dw.cache
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    q = torch.zeros((0, 8, 64), dtype=torch.bfloat16, device="cuda")
    out = nat.attention(c, q, dw.block_tables[:0], z, z, 1, 0.1, dw.workspace)
    assert out.shape == (0, 8, 64)
    nat.append(c, q[:, :2].contiguous(), q[:, :2].contiguous(), torch.zeros(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_wait_timeout_reports_and_recovers(dtype):
    """The device timeout path, made to run out without a fault: a wait
    limit of 200 us and a hold flag that nothing sets.  The producer's bounded
    wait on the flag gives up, raises PKV_DEVERR_TIMEOUT and the abort flag,
    and every role of every CTA winds down (no copy in flight, TMEM freed):
    the call returns and the context stays usable.  After the workspace is
    zeroed again the same workspace gives oracle parity."""
    w = wl.make_workload("to", context_lens=[300, 77, 1000, 40], q_lens=[1, 1, 1, 1], num_q_heads=32,
                         num_kv_heads=8, head_dim=128, kv_dtype=dtype, seed=95)
    dw = DeviceWorkload(w)
    dw.prefill()
    dw.append_step()
    hold = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        nat.debug_set_wait_limit(200_000, hold)
        dw.attend()
        torch.cuda.synchronize()
    finally:
        nat.debug_set_wait_limit(0, None)
    assert nat.read_device_error(dw.workspace) == nat.DEVERR_TIMEOUT
    nat.workspace_init(dw.workspace)
    out = dw.attend()
    kc, vc = oracle.build_cache(w)
    ref, _ = oracle.attend(w, kc, vc)
    assert_attention_close(out_bits(out), ref, "after a timeout")
    assert dw.errors() == (0, 0)

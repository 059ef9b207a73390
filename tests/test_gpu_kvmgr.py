"""The block manager driving the GPU path: conversations whose turns share a
system prompt get their block tables and slots from pkv_kvmgr_* (prefix
blocks reused through the radix tree, K/V of the shared prefix written once),
the kernels append and attend through them, and the result matches the
oracle run on the same slots and tables.  A fork whose child writes into the
shared partially filled block exercises copy-on-write (pkv_copy_blocks on
the device, the same copy on the oracle's cache)."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import _native as nat
from paged_kv_decode_14_gb300 import workloads as wl
from gpu_helpers import assert_attention_close, caches_equal, out_bits

pytestmark = pytest.mark.gpu

Hq, Hkv, D = 32, 8, 64


def _kv_rows(rng, n):
    return (wl.bf16_bits(rng.standard_normal((n, Hkv, D), dtype=np.float32)),
            wl.bf16_bits(rng.standard_normal((n, Hkv, D), dtype=np.float32)))


class _Mirror:
    """The device cache and an oracle cache, written through the same slots."""

    def __init__(self, num_blocks, dtype):
        self.w = wl.make_workload("m", context_lens=[1], q_lens=[1], num_q_heads=Hq, num_kv_heads=Hkv,
                                  head_dim=D, kv_dtype=dtype, num_blocks=num_blocks, seed=1)
        self.nb = num_blocks
        self.dtype = dtype
        ks = vs = None
        if dtype == "fp8":
            rng = np.random.default_rng(5)
            self.ks = rng.uniform(0.002, 0.01, (num_blocks, Hkv)).astype(np.float32)
            self.vs = rng.uniform(0.002, 0.01, (num_blocks, Hkv)).astype(np.float32)
            ks, vs = torch.from_numpy(self.ks).cuda(), torch.from_numpy(self.vs).cuda()
        else:
            self.ks = self.vs = None
        self.cache = nat.PagedKVCache(num_blocks, Hkv, D, dtype, k_scales=ks, v_scales=vs)
        fill = int(wl.FP8_NAN) if dtype == "fp8" else int(np.int16(wl.BF16_NAN.view(np.int16)))
        (self.cache.k.view(torch.uint8) if dtype == "fp8" else self.cache.k.view(torch.int16)).fill_(fill)
        (self.cache.v.view(torch.uint8) if dtype == "fp8" else self.cache.v.view(torch.int16)).fill_(fill)
        self.kc, self.vc = self.w.empty_cache(), self.w.empty_cache()
        self.kd = oracle.KV_FP8 if dtype == "fp8" else oracle.KV_BF16

    def append(self, k, v, slots):
        slots = np.asarray(slots, dtype=np.int64)
        oracle.paged_kv_append(self.kd, self.kc, self.vc, self.ks, self.vs, self.nb, Hkv, D, k, v, slots)
        kt = torch.from_numpy(k.view(np.int16)).cuda().view(torch.bfloat16)
        vt = torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16)
        nat.append(self.cache, kt, vt, torch.from_numpy(slots).cuda())

    def copy(self, src, dst):
        e = 1 if self.dtype == "fp8" else 2
        page = Hkv * 16 * D
        for c in (self.kc, self.vc):
            c[dst * page:(dst + 1) * page] = c[src * page:(src + 1) * page]
        if self.ks is not None:
            self.ks[dst] = self.ks[src]
            self.vs[dst] = self.vs[src]
        nat.copy_blocks(self.cache, torch.tensor([[src, dst]], dtype=torch.int32).cuda())
        del e

    def attend_and_check(self, mgr, seqs, q, what):
        mb = 64
        bt, lens = mgr.tables(seqs, mb)
        ql = np.ones(len(seqs), np.int32)
        ref, _ = oracle.paged_attention(self.kd, self.kc, self.vc, self.ks, self.vs, self.nb, Hkv, D, q, Hq, bt,
                                        lens, ql, 0.125)
        dev = "cuda"
        ws = nat.make_workspace(len(seqs), Hq, Hkv, D, 1)
        qt = torch.from_numpy(q.view(np.int16)).to(dev).view(torch.bfloat16)
        out = nat.attention(self.cache, qt, torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev),
                            torch.from_numpy(ql).to(dev), 1, 0.125, ws)
        torch.cuda.synchronize()
        assert_attention_close(out_bits(out), ref, what)
        assert nat.read_device_error(ws) == 0
        gk = (self.cache.k.view(torch.uint8) if self.dtype == "fp8" else self.cache.k.view(torch.int16)).cpu().numpy()
        gk = gk.reshape(-1) if self.dtype == "fp8" else gk.reshape(-1).view(np.uint16)
        assert caches_equal(gk, self.kc, self.dtype == "fp8")


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_conversations_through_the_block_manager(dtype):
    rng = np.random.default_rng(31)
    mgr = nat.KVManager(400)
    mirror = _Mirror(400, dtype)
    system = rng.integers(0, 1000, 700).tolist()                     # 43 full blocks + 12 tokens
    seqs = []
    for t in range(4):                                               # 4 turns of one conversation
        prompt = system + rng.integers(0, 1000, int(rng.integers(30, 200))).tolist()
        cached, slots = mgr.add_sequence(t, prompt)
        assert cached == (0 if t == 0 else 16 * (len(system) // 16))  # the system prompt's full blocks
        k, v = _kv_rows(rng, len(slots))
        mirror.append(k, v, slots)                                   # only the uncached part is written
        mgr.commit(t)
        seqs.append(t)
    bt, _ = mgr.tables(seqs, 64)
    assert all((bt[t, :43] == bt[0, :43]).all() for t in range(4))   # one copy of the shared prefix
    # a decode step: one new token per turn, then attention over all four
    for t in seqs:
        slots, copy = mgr.append(t, [int(rng.integers(0, 1000))])
        assert copy is None
        k, v = _kv_rows(rng, 1)
        mirror.append(k, v, slots)
    q = wl.bf16_bits(rng.standard_normal((4, Hq, D), dtype=np.float32))
    mirror.attend_and_check(mgr, seqs, q, f"{dtype} conversations")
    # fork turn 0 mid-block: both branches write a token; the child copies the shared block first
    while mgr.tables([0], 64)[1][0] % 16 == 0:
        slots, _ = mgr.append(0, [3])
        k, v = _kv_rows(rng, 1)
        mirror.append(k, v, slots)
    mgr.fork(0, 10)
    slots_c, copy = mgr.append(10, [5])
    assert copy is not None
    mirror.copy(*copy)
    k, v = _kv_rows(rng, 1)
    mirror.append(k, v, slots_c)
    slots_p, copy_p = mgr.append(0, [6])
    assert copy_p is None and slots_p[0] // 16 == copy[0]           # the parent keeps writing the original
    k, v = _kv_rows(rng, 1)
    mirror.append(k, v, slots_p)
    q2 = wl.bf16_bits(rng.standard_normal((2, Hq, D), dtype=np.float32))
    mirror.attend_and_check(mgr, [0, 10], q2, f"{dtype} fork")

"""Host-side checks that need no GPU: the C-ABI library builds for sm_103a,
loads, and exports every entry point include/pagedkv.h declares; the binding
refuses to run without it; the workload generator's structure."""

import ctypes
import os
import re
import shutil

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def declared_symbols():
    """Every entry point any header under include/ declares."""
    syms = []
    for n in sorted(os.listdir(INCLUDE)):
        if n.endswith(".h"):
            src = open(os.path.join(INCLUDE, n)).read()
            syms += re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", src)
    return syms


def _built_lib():
    from paged_kv_decode_14_gb300 import build as b
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        if not os.path.exists(b.LIB):
            pytest.skip("no nvcc and no prebuilt library")
        return b.LIB
    return b.build()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("pkv_paged_kv_append", "pkv_paged_attention", "pkv_attention_workspace_size",
              "pkv_workspace_init", "pkv_read_device_error", "pkv_status_string", "pkv_version",
              "pkv_kvmgr_create", "pkv_kvmgr_add_sequence", "pkv_kvmgr_append", "pkv_kvmgr_tables",
              "pkv_copy_blocks"):
        assert s in syms


def test_library_exports_every_declared_symbol():
    path = _built_lib()
    lib = ctypes.CDLL(path)
    for s in declared_symbols():
        assert hasattr(lib, s), f"{s} declared in pagedkv.h but not exported"
    lib.pkv_status_string.restype = ctypes.c_char_p
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(3).startswith(b"workspace")
    # no GPU calls here: only the pure host helpers
    lib.pkv_attention_workspace_size.restype = ctypes.c_size_t
    assert lib.pkv_attention_workspace_size(4, 8, 3, 64, 1, 16) == 0   # Hq % Hkv != 0


def test_exports_are_only_the_abi():
    """The shared object exports the pkv_* ABI and nothing of its internals."""
    path = _built_lib()
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    names = [ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln]
    pkv = [n for n in names if n.startswith("pkv_")]
    assert sorted(pkv) == sorted(set(declared_symbols()))


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from paged_kv_decode_14_gb300 import _native as nat
    monkeypatch.setattr(nat, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(nat, "_lib", None)
    with pytest.raises(RuntimeError, match="libpagedkv.so not found"):
        nat.lib()


def test_workload_structure():
    from paged_kv_decode_14_gb300 import workloads as wl
    w = wl.prefix_reuse_b32_d64()
    assert w.num_seqs == 32 and w.head_dim == 64
    # turns of a conversation share their prefix blocks
    for c in range(8):
        rows = w.block_tables[4 * c:4 * c + 4]
        L = w.context_lens[4 * c:4 * c + 4]
        shared = 0
        while all(rows[t, shared] == rows[0, shared] for t in range(4)) and shared < min((L - 1) // 16):
            shared += 1
        assert 32 <= shared <= 96
    # every slot lies in the block its sequence's table names
    slots = np.concatenate([w.prefill_slots, w.slots])
    assert len(set(slots.tolist())) == len(slots)          # no duplicate slot
    assert np.all(slots // 16 < w.num_blocks)
    w2 = wl.decode_b32_d128()
    assert w2.num_blocks == 5000 and np.all((w2.context_lens >= 256) & (w2.context_lens <= 2048))
    assert 100e6 < w2.kv_bytes() < 220e6
    # seeded: the same config twice gives the same inputs
    assert np.array_equal(wl.decode_b32_d128().q, w2.q)


def test_fp8_scales_are_absmax_over_448():
    from paged_kv_decode_14_gb300 import workloads as wl
    w = wl.make_workload("f", context_lens=[40, 7], q_lens=[1, 1], num_q_heads=4, num_kv_heads=2,
                         head_dim=64, kv_dtype="fp8", seed=3, outlier_p=0.01)
    allk = wl.bf16_to_f32(np.concatenate([w.prefill_k, w.k_new]))
    slots = np.concatenate([w.prefill_slots, w.slots])
    for blk in set((slots // 16).tolist()):
        sel = slots // 16 == blk
        for g in range(2):
            exp = np.float32(np.abs(allk[sel, g]).max()) / np.float32(448.0)
            assert w.k_scales[blk, g] == exp


def test_causal_flops_counts_every_visible_pair():
    """The prefill metric's FLOP count: 4 * D * Hq per (query, visible key),
    against a brute-force count of the pairs the definition makes visible
    (query i of sequence b sees positions 0 .. L_b - Q_b + i)."""
    from paged_kv_decode_14_gb300 import workloads as wl
    w = wl.make_workload("flops", context_lens=[1, 17, 40, 300, 0], q_lens=[1, 5, 40, 128, 0], num_q_heads=8,
                         num_kv_heads=2, head_dim=64, seed=3)
    pairs = 0
    for L, Q in zip(w.context_lens.tolist(), w.q_lens.tolist()):
        for i in range(Q):
            pairs += sum(1 for j in range(L) if j <= L - Q + i)
    assert wl.causal_flops(w) == 4 * 64 * 8 * pairs

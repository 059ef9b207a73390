"""Pins for the CPU oracle: checks against things other than the oracle itself.

* e4m3: torch's float8_e4m3fn decode of all 256 codes, a brute-force
  nearest-code search over every bf16 bit pattern at several scales, torch's
  RNE cast inside the finite range, and the OCP landmark codes
  (tests/golden/e4m3fn_landmarks.txt).
* bf16 rounding: brute force over neighbours and torch's fp32 -> bf16 cast.
* cache layout: a numpy reshape/transpose statement of the page layout.
* attention: torch.nn.functional.scaled_dot_product_attention in fp64 on the
  gathered context (paged == dense, the inferd "Paged KV equivalence" gate),
  closed forms (length-1 context, zero query, equal keys, dominant logit, the
  hand-worked two-token example) and invariants (block permutation, prefix
  sharing).
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_14_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------- e4m3

def _all_codes_values():
    return np.array([oracle.e4m3_decode(c) for c in range(256)], dtype=np.float64)


def test_e4m3_decode_matches_torch_all_codes():
    mine = _all_codes_values()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_m, nan_r = np.isnan(mine), np.isnan(ref)
    assert np.array_equal(nan_m, nan_r)
    assert nan_m.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(mine[~nan_m], ref[~nan_r])
    assert np.array_equal(np.signbit(mine[~nan_m]), np.signbit(ref[~nan_r]))


def test_e4m3_golden_landmarks():
    with open(os.path.join(GOLDEN, "e4m3fn_landmarks.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for code_s, val_s in rows:
        code = int(code_s, 16)
        v = oracle.e4m3_decode(code)
        if val_s == "nan":
            assert math.isnan(v)
            continue
        exp = float(val_s)
        assert v == exp and math.copysign(1, v) == math.copysign(1, exp), (code_s, v, exp)
        # the encoder maps each landmark value back to its code
        assert oracle.e4m3_encode(exp) == code


def _brute_force_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest finite code of the same sign; ties to the even code; |x| > 448 -> 448."""
    vals = _all_codes_values()
    pos_codes = np.array([c for c in range(128) if c != 0x7F])
    pos_vals = vals[pos_codes]
    x = x.astype(np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    a = np.minimum(a, 448.0)
    for s in range(0, a.size, 8192):
        blk = a[s:s + 8192, None]
        d = np.abs(blk - pos_vals[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        # among ties pick the even code (mantissa LSB 0)
        even = cand & ((pos_codes[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        out[s:s + 8192] = pos_codes[pick]
    out = np.where(sign, out | 0x80, out).astype(np.uint8)
    out = np.where(nan, np.where(sign, 0xFF, 0x7F), out).astype(np.uint8)
    return out


@pytest.mark.parametrize("scale", [1.0, 0.5, 1.0 / 448.0, 3.7, 1e-3, 2.0 ** -130, 0.0826])
def test_e4m3_encode_brute_force_all_bf16(scale):
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << np.uint32(16)).view(np.float32)
    with np.errstate(all="ignore"):
        quot = (x / np.float32(scale)).astype(np.float32)   # one fp32 IEEE division
    mine = oracle.e4m3_encode_array(quot)
    ref = _brute_force_e4m3(quot)
    isnan = np.isnan(quot)
    assert np.array_equal(mine[~isnan], ref[~isnan])
    # NaN inputs: any NaN code is correct (both S.1111.111 patterns)
    assert np.all((mine[isnan] & 0x7F) == 0x7F)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * s
                        for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    mine = oracle.e4m3_encode_array(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_e4m3_saturation_and_specials():
    assert oracle.e4m3_encode(449.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00           # tie -> even (0)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02       # tie -> even (2)
    assert oracle.e4m3_encode(-2.0 ** -11) == 0x80          # rounds to -0


# ------------------------------------------------------------------------- bf16

def _bf16_neighbours_round(x: float) -> int:
    """Brute force: the two bf16 values around x, nearest wins, ties to even bits."""
    f = np.float32(x)  # a starting point near x
    b = int(np.array([f], np.float32).view(np.uint32)[0] >> 16)
    best = None
    for cand in range(max(0, b - 2), min(0xFFFF, b + 3)):
        for sgn in (0, 0x8000):
            c = (cand & 0x7FFF) | sgn
            v = float((np.array([c << 16], np.uint32)).view(np.float32)[0])
            if math.isnan(v) or math.isinf(v):
                continue
            d = abs(v - x)
            key = (d, c & 1)
            if best is None or key < best[0]:
                best = (key, c)
    return best[1]


def test_bf16_round_brute_force():
    rng = np.random.default_rng(5)
    xs = list(rng.standard_normal(3000) * np.exp(rng.uniform(-30, 30, 3000)))
    # exact ties: midpoints between adjacent bf16 values
    for base in (1.0, 1.0 + 2 ** -7, 3.0, 1e-20, 7e10):
        b = int(np.array([base], np.float32).view(np.uint32)[0] >> 16)
        lo = float(np.array([b << 16], np.uint32).view(np.float32)[0])
        hi = float(np.array([(b + 1) << 16], np.uint32).view(np.float32)[0])
        xs += [(lo + hi) / 2, -(lo + hi) / 2]
    for x in xs:
        assert oracle.bf16_round(x) == _bf16_neighbours_round(x), x


def test_bf16_round_matches_torch_on_floats():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(50000) * 10.0).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([oracle.bf16_round(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(mine, ref)
    assert oracle.bf16_round(float("inf")) == 0x7F80
    assert oracle.bf16_round(3.5e38) == 0x7F80
    assert oracle.bf16_round(-0.0) == 0x8000


# ------------------------------------------------------------------------- layout

def np_page_to_dense(page: np.ndarray, head_dim: int, elem_bytes: int) -> np.ndarray:
    """Page [16/8][D/C][8][C] -> [16 tokens][D] (numpy restatement of the layout)."""
    C = 16 // elem_bytes
    return page.reshape(2, head_dim // C, 8, C).transpose(0, 2, 1, 3).reshape(16, head_dim)


def np_gather(cache: np.ndarray, table_row, L, g, num_kv_heads, head_dim, elem_bytes) -> np.ndarray:
    """Dense [L, D] rows of kv-head g for one sequence, via the numpy layout statement."""
    pages = cache.reshape(-1, num_kv_heads, 16 * head_dim)
    nb = (L + 15) // 16
    rows = [np_page_to_dense(pages[table_row[j], g], head_dim, elem_bytes) for j in range(nb)]
    return np.concatenate(rows, axis=0)[:L] if rows else np.zeros((0, head_dim), cache.dtype)


@pytest.mark.parametrize("D,e", [(64, 2), (128, 2), (64, 1), (128, 1), (8, 2), (16, 1)])
def test_cache_index_matches_numpy_layout(D, e):
    Hkv, NB = 3, 4
    n = NB * Hkv * 16 * D
    ids = np.arange(n, dtype=np.int64)
    pages = ids.reshape(NB, Hkv, 16 * D)
    for blk in range(NB):
        for g in range(Hkv):
            dense = np_page_to_dense(pages[blk, g], D, e)
            for off in (0, 1, 7, 8, 15):
                for d in (0, 1, D // 2, D - 1):
                    assert oracle.cache_index(blk, g, off, d, Hkv, D, e) == dense[off, d]


# ------------------------------------------------------------------------- append

def test_append_bf16_matches_numpy_scatter():
    w = wl.make_workload("t", context_lens=[5, 40, 17], q_lens=[1, 1, 1], num_q_heads=4,
                         num_kv_heads=2, head_dim=64, seed=3)
    kc, vc = oracle.build_cache(w)
    # numpy statement: scatter each token into its dense page row
    ek = w.empty_cache().reshape(w.num_blocks, 2, 16 * 64).copy()
    allk = np.concatenate([w.prefill_k, w.k_new])
    slots = np.concatenate([w.prefill_slots, w.slots])
    dense = {}
    for t, s in enumerate(slots):
        blk, off = divmod(int(s), 16)
        for g in range(2):
            pg = dense.setdefault((blk, g), np_page_to_dense(ek[blk, g].copy(), 64, 2))
            pg[off] = allk[t, g]
    for (blk, g), pg in dense.items():
        C = 8
        ek[blk, g] = pg.reshape(2, 8, 64 // C, C).transpose(0, 2, 1, 3).reshape(-1)
    assert np.array_equal(kc.view(np.uint16), ek.reshape(-1))


def test_append_skips_negative_and_counts_out_of_range():
    kc = np.full(2 * 1 * 16 * 64, wl.BF16_NAN, np.uint16)
    vc = kc.copy()
    k = np.arange(3 * 64, dtype=np.uint16).reshape(3, 1, 64)
    bad = oracle.paged_kv_append(0, kc, vc, None, None, 2, 1, 64, k, k, np.array([-1, 33, 5]))
    assert bad == 1
    d = np_page_to_dense(kc.reshape(2, 16 * 64)[0], 64, 2)
    assert np.array_equal(d[5], k[2, 0])
    assert np.all(kc.reshape(2, -1)[1] == wl.BF16_NAN)   # slot 33 (block 2) not written


def test_append_fp8_matches_brute_force():
    w = wl.make_workload("t8", context_lens=[30, 70], q_lens=[1, 2], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, kv_dtype="fp8", seed=9, outlier_p=0.01)
    kc, vc = oracle.build_cache(w)
    allk = np.concatenate([w.prefill_k, w.k_new])
    slots = np.concatenate([w.prefill_slots, w.slots])
    pages = kc.reshape(w.num_blocks, 2, 16 * 128)
    for t in range(0, len(slots), 7):
        blk, off = divmod(int(slots[t]), 16)
        for g in range(2):
            src = wl.bf16_to_f32(allk[t, g])
            quot = (src / np.float32(w.k_scales[blk, g])).astype(np.float32)
            exp = _brute_force_e4m3(quot)
            got = np_page_to_dense(pages[blk, g], 128, 1)[off]
            assert np.array_equal(got, exp)


# ------------------------------------------------------------------------- attention

def dense_sdpa_reference(w, kc, vc):
    """torch SDPA in fp64 on K/V gathered with the numpy layout statement."""
    e = w.elem_bytes
    G = w.num_q_heads // w.num_kv_heads
    qf = torch.from_numpy(wl.bf16_to_f32(w.q).astype(np.float64))
    out = torch.zeros(qf.shape, dtype=torch.float64)
    qoff = 0
    for b in range(w.num_seqs):
        L, Q = int(w.context_lens[b]), int(w.q_lens[b])
        ks, vs = [], []
        for g in range(w.num_kv_heads):
            kk = np_gather(kc, w.block_tables[b], L, g, w.num_kv_heads, w.head_dim, e)
            vv = np_gather(vc, w.block_tables[b], L, g, w.num_kv_heads, w.head_dim, e)
            if w.kv_dtype == "fp8":
                tab = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
                blk = w.block_tables[b, np.arange(L) // 16]
                kk = tab[kk] * w.k_scales[blk, g][:, None].astype(np.float64)
                vv = tab[vv] * w.v_scales[blk, g][:, None].astype(np.float64)
            else:
                kk, vv = wl.bf16_to_f32(kk).astype(np.float64), wl.bf16_to_f32(vv).astype(np.float64)
            ks.append(torch.from_numpy(kk))
            vs.append(torch.from_numpy(vv))
        K = torch.stack(ks).repeat_interleave(G, dim=0)      # [Hq, L, D]
        V = torch.stack(vs).repeat_interleave(G, dim=0)
        qb = qf[qoff:qoff + Q].transpose(0, 1)               # [Hq, Q, D]
        pos = torch.arange(L)[None, :]
        lim = (L - Q + torch.arange(Q))[:, None]
        mask = pos <= lim                                    # [Q, L]
        o = torch.nn.functional.scaled_dot_product_attention(qb, K, V, attn_mask=mask, scale=float(w.scale))
        out[qoff:qoff + Q] = o.transpose(0, 1)
        qoff += Q
    return out.numpy()


@pytest.mark.parametrize("case", ["tiny", "verify", "prefix", "fp8", "d128", "prefill"])
def test_attention_equals_dense_sdpa(case):
    if case == "tiny":
        w = wl.tiny_decode()
    elif case == "verify":
        w = wl.make_workload("v", context_lens=[9, 40, 77], q_lens=[5, 3, 8], num_q_heads=8,
                             num_kv_heads=2, head_dim=64, seed=21)
    elif case == "prefix":
        w = wl.make_workload("p", context_lens=[48, 70, 33, 90], q_lens=[1, 1, 1, 1], num_q_heads=8,
                             num_kv_heads=4, head_dim=64, seed=22, shared_prefix=[(0, 3, 32)])
    elif case == "fp8":
        w = wl.make_workload("f", context_lens=[20, 130, 1], q_lens=[1, 2, 1], num_q_heads=8,
                             num_kv_heads=2, head_dim=128, kv_dtype="fp8", seed=23, outlier_p=0.01)
    elif case == "d128":
        w = wl.make_workload("d", context_lens=[100, 3], q_lens=[1, 1], num_q_heads=8,
                             num_kv_heads=1, head_dim=128, seed=24)
    else:
        # whole prompts: every token is a query, the first one sees only itself
        w = wl.make_workload("c", context_lens=[17, 33, 1], q_lens=[17, 33, 1], num_q_heads=8,
                             num_kv_heads=2, head_dim=64, seed=25)
    kc, vc = oracle.build_cache(w)
    out, outb = oracle.attend(w, kc, vc)
    ref = dense_sdpa_reference(w, kc, vc)
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    # bf16 output is the single rounding of the fp64 value
    rb = np.array([oracle.bf16_round(v) for v in out.ravel()[:4096]], dtype=np.uint16)
    assert np.array_equal(outb.ravel()[:4096], rb)


def _single_seq(L, q_vals=None, k_vals=None, v_vals=None, D=64, Hq=4, Hkv=1, seed=0):
    w = wl.make_workload("s", context_lens=[L], q_lens=[1], num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, seed=seed)
    if q_vals is not None:
        w.q[:] = q_vals
    if k_vals is not None:
        w.prefill_k[:] = k_vals
        w.k_new[:] = k_vals
    if v_vals is not None:
        w.prefill_v[:] = v_vals
        w.v_new[:] = v_vals
    return w


def test_closed_form_length_one_context_returns_v():
    w = _single_seq(1, seed=31)
    kc, vc = oracle.build_cache(w)
    out, outb = oracle.attend(w, kc, vc)
    for h in range(4):
        assert np.array_equal(outb[0, h], w.v_new[0, 0])          # bitwise: out = v0
        assert np.array_equal(out[0, h], wl.bf16_to_f32(w.v_new[0, 0]).astype(np.float64))


def test_closed_form_zero_query_is_mean_of_v():
    w = _single_seq(37, q_vals=0, seed=32)
    kc, vc = oracle.build_cache(w)
    out, _ = oracle.attend(w, kc, vc)
    allv = wl.bf16_to_f32(np.concatenate([w.prefill_v, w.v_new])[:, 0]).astype(np.float64)
    assert np.allclose(out[0, 0], allv.mean(axis=0), rtol=0, atol=1e-13)


def test_closed_form_equal_keys_is_mean_of_v():
    w = _single_seq(50, seed=33)
    w.prefill_k[:] = w.prefill_k[0]
    w.k_new[:] = w.prefill_k[0]
    kc, vc = oracle.build_cache(w)
    out, _ = oracle.attend(w, kc, vc)
    allv = wl.bf16_to_f32(np.concatenate([w.prefill_v, w.v_new])[:, 0]).astype(np.float64)
    assert np.allclose(out[0, 2], allv.mean(axis=0), rtol=0, atol=1e-13)


def test_closed_form_dominant_logit_selects_v():
    w = _single_seq(40, seed=34)
    allk = np.concatenate([w.prefill_k, w.k_new])
    j_star = 17
    w.q[0, :] = allk[j_star, 0]
    w.scale = 64.0    # q.k_j* / |...| dominates every other logit by a wide margin
    kc, vc = oracle.build_cache(w)
    out, _ = oracle.attend(w, kc, vc)
    allv = wl.bf16_to_f32(np.concatenate([w.prefill_v, w.v_new])[:, 0]).astype(np.float64)
    assert np.allclose(out[0, 0], allv[j_star], rtol=0, atol=1e-9)


def test_golden_two_token_example():
    D = 8
    kc = np.full(1 * 1 * 16 * D, wl.BF16_NAN, np.uint16)
    vc = kc.copy()
    one, two = 0x3F80, 0x4000
    k = np.zeros((2, 1, D), np.uint16)
    v = np.zeros((2, 1, D), np.uint16)
    k[1, 0, 0] = one
    v[1, 0, 0], v[1, 0, 1] = one, two
    oracle.paged_kv_append(0, kc, vc, None, None, 1, 1, D, k, v, np.array([0, 1]))
    q = np.zeros((1, 1, D), np.uint16)
    q[0, 0, 0] = one
    out, _ = oracle.paged_attention(0, kc, vc, None, None, 1, 1, D, q, 1, np.array([[0]]),
                                    np.array([2]), np.array([1]), 1.0)
    with open(os.path.join(GOLDEN, "two_token_attention.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for d_s, v_s in rows:
        assert abs(out[0, 0, int(d_s)] - float(v_s)) < 1e-15


def test_invariant_block_permutation():
    w = wl.make_workload("perm", context_lens=[70, 33, 128], q_lens=[1, 3, 2], num_q_heads=8,
                         num_kv_heads=2, head_dim=64, seed=41)
    kc, vc = oracle.build_cache(w)
    out, _ = oracle.attend(w, kc, vc)
    rng = np.random.default_rng(1)
    perm = rng.permutation(w.num_blocks)          # old block -> new block
    pages_k = kc.reshape(w.num_blocks, -1)
    pages_v = vc.reshape(w.num_blocks, -1)
    nk, nv = np.empty_like(pages_k), np.empty_like(pages_v)
    nk[perm], nv[perm] = pages_k, pages_v
    w.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, _ = oracle.attend(w, nk.reshape(-1), nv.reshape(-1))
    assert np.array_equal(out, out2)


def test_invariant_shared_prefix_equals_private_copies():
    w = wl.make_workload("sh", context_lens=[64, 80, 50], q_lens=[1, 1, 1], num_q_heads=8,
                         num_kv_heads=2, head_dim=64, seed=42, shared_prefix=[(0, 3, 48)],
                         num_blocks=40)
    kc, vc = oracle.build_cache(w)
    out, _ = oracle.attend(w, kc, vc)
    # copy the shared blocks of sequences 1 and 2 into fresh private blocks
    used = set(int(x) for x in w.block_tables[w.block_tables >= 0])
    free = [b for b in range(w.num_blocks) if b not in used]
    pk, pv = kc.reshape(w.num_blocks, -1).copy(), vc.reshape(w.num_blocks, -1).copy()
    for s in (1, 2):
        for j in range(3):
            nb = free.pop()
            pk[nb], pv[nb] = pk[w.block_tables[s, j]], pv[w.block_tables[s, j]]
            w.block_tables[s, j] = nb
    out2, _ = oracle.attend(w, pk.reshape(-1), pv.reshape(-1))
    assert np.array_equal(out, out2)


def test_oracle_reports_bad_inputs():
    w = wl.make_workload("bad", context_lens=[20], q_lens=[1], num_q_heads=2, num_kv_heads=1,
                         head_dim=64, seed=43)
    kc, vc = oracle.build_cache(w)
    w.q_lens = np.array([25], np.int32)
    w.q = np.zeros((25, 2, 64), np.uint16)
    with pytest.raises(ValueError, match="status 2"):
        oracle.attend(w, kc, vc)
    w.q_lens = np.array([1], np.int32)
    w.q = np.zeros((1, 2, 64), np.uint16)
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 1] = w.num_blocks + 5
    with pytest.raises(ValueError, match="status 3"):
        oracle.attend(w, kc, vc)


# ------------------------------------------------------------------------- RoPE, FP8 scales

def test_rope_golden_hand_worked():
    for ln in open(os.path.join(GOLDEN, "rope_example.txt")):
        if ln.startswith("#") or not ln.strip():
            continue
        f = ln.split()
        theta, pos = float(f[0]), int(f[1])
        x = np.array([int(v, 16) for v in f[2:6]], np.uint16).reshape(1, 1, 4)
        want = np.array([int(v, 16) for v in f[6:10]], np.uint16)
        assert oracle.rope(x, [pos], theta).reshape(-1).tolist() == want.tolist()


def _bf16_rows(rng, shape):
    return wl.bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def test_rope_invariants():
    """Position 0 is the identity; each (i, i + D/2) pair keeps its norm; a
    rotation by p1 then by p2 equals one by p1 + p2; and scores of rotated
    rows depend only on the positions' difference (up to bf16 rounding)."""
    rng = np.random.default_rng(11)
    T, H, D = 6, 3, 64
    x = _bf16_rows(rng, (T, H, D))
    assert np.array_equal(oracle.rope(x, np.zeros(T, np.int32), 1e4), x)
    pos = rng.integers(0, 40000, T).astype(np.int32)
    y = oracle.rope(x, pos, 1e4)
    fx, fy = wl.bf16_to_f32(x).astype(np.float64), wl.bf16_to_f32(y).astype(np.float64)
    nx = fx[..., :D // 2] ** 2 + fx[..., D // 2:] ** 2
    ny = fy[..., :D // 2] ** 2 + fy[..., D // 2:] ** 2
    assert np.all(np.abs(ny - nx) <= 2.0 ** -6 * nx + 1e-30)
    p1, p2 = rng.integers(0, 3000, T).astype(np.int32), rng.integers(0, 3000, T).astype(np.int32)
    two = wl.bf16_to_f32(oracle.rope(oracle.rope(x, p1, 1e4), p2, 1e4)).astype(np.float64)
    one = wl.bf16_to_f32(oracle.rope(x, p1 + p2, 1e4)).astype(np.float64)
    assert np.max(np.abs(two - one)) <= 2.0 ** -6 * np.max(np.abs(one))
    q = _bf16_rows(rng, (1, 1, D))
    k = _bf16_rows(rng, (1, 1, D))
    def score(a, b):
        qa = wl.bf16_to_f32(oracle.rope(q, [a], 1e4)).astype(np.float64).reshape(-1)
        kb = wl.bf16_to_f32(oracle.rope(k, [b], 1e4)).astype(np.float64).reshape(-1)
        return float(qa @ kb)
    base = score(100, 37)
    for shift in (1, 50, 9000):
        assert abs(score(100 + shift, 37 + shift) - base) <= 0.05 * (1.0 + abs(base))


def test_fp8_autoscale_recipe():
    """Blocks this append starts get absmax / 448 (fp32) over the call's values
    in that block and head (NaN ignored, 1.0 if all zero) -- the same recipe
    as the input generator's, computed here with numpy; others keep theirs."""
    rng = np.random.default_rng(12)
    Hkv, D, NB = 2, 64, 6
    T = 40                                                     # block 1: offsets 0..15, block 2: 0..15, block 4: 0..7
    slots = np.concatenate([16 + np.arange(16), 32 + np.arange(16), 64 + np.arange(8)]).astype(np.int64)
    k = _bf16_rows(rng, (T, Hkv, D))
    v = _bf16_rows(rng, (T, Hkv, D))
    v[16:32, 1] = 0                                            # block 2, head 1: all zero V
    k[3, 0, 5] = np.uint16(0x7FC0)                             # a NaN in block 1, head 0
    extra = np.array([[5 * 16 + 3]], np.int64).reshape(-1)     # block 5 continued (offset 3): keeps its scale
    slots = np.concatenate([slots, extra])
    k = np.concatenate([k, _bf16_rows(rng, (1, Hkv, D))])
    v = np.concatenate([v, _bf16_rows(rng, (1, Hkv, D))])
    ks = np.full((NB, Hkv), 7.0, np.float32)
    vs = np.full((NB, Hkv), 7.0, np.float32)
    oracle.fp8_autoscale(k, v, slots, NB, ks, vs)
    fk, fv = wl.bf16_to_f32(k), wl.bf16_to_f32(v)
    for blk, rows in ((1, slice(0, 16)), (2, slice(16, 32)), (4, slice(32, 40))):
        for g in range(Hkv):
            ak = np.nanmax(np.abs(fk[rows, g]))
            av = np.nanmax(np.abs(fv[rows, g]))
            assert ks[blk, g] == (np.float32(ak) / np.float32(448.0) if ak > 0 else np.float32(1.0))
            assert vs[blk, g] == (np.float32(av) / np.float32(448.0) if av > 0 else np.float32(1.0))
    assert vs[2, 1] == 1.0
    assert np.all(ks[[0, 3, 5]] == 7.0) and np.all(vs[[0, 3, 5]] == 7.0)

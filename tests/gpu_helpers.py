"""Shared helpers of the GPU parity tests (no test functions here)."""

import functools

import numpy as np
import torch

import oracle
from paged_kv_decode_14_gb300 import workloads as wl

# Attention tolerance: |gpu - oracle_fp64| <= ATOL + RTOL * |oracle_fp64| element-wise
# (max-abs 2e-3 and max-rel 1e-2 of the problem statement, read as allclose).
ATOL, RTOL = 2e-3, 1e-2


def to_f64(bits: np.ndarray) -> np.ndarray:
    return wl.bf16_to_f32(bits).astype(np.float64)


def out_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_attention_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str = "", nan_aware: bool = False):
    """Element-wise tolerance check.  By default any NaN in the GPU output
    fails.  With nan_aware, an element must be NaN on the GPU exactly where
    the oracle's is (a NaN stored in the cache propagates), and the others
    must be within the tolerance."""
    g = to_f64(gpu_bits)
    if nan_aware:
        gn, rn = np.isnan(g), np.isnan(ref)
        if not np.array_equal(gn, rn):
            i = np.argwhere(gn != rn)[0]
            raise AssertionError(f"{what}: NaN pattern differs ({int(gn.sum())} NaN on the GPU, "
                                 f"{int(rn.sum())} in the oracle); first at {tuple(i)}")
        g = np.where(gn, 0.0, g)
        ref = np.where(rn, 0.0, ref)
    else:
        assert not np.isnan(g).any(), f"{what}: NaN in GPU output"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(i)}: "
                             f"gpu {g[tuple(i)]} oracle {ref[tuple(i)]}; max abs err {err.max()}")
    return float(err.max())


def caches_equal(a: np.ndarray, b: np.ndarray, fp8: bool) -> bool:
    """Bitwise cache equality; NaN codes of E4M3 (both signs) count as equal."""
    if a.shape != b.shape:
        return False
    if fp8:
        nan_a, nan_b = (a & 0x7F) == 0x7F, (b & 0x7F) == 0x7F
        return bool(np.array_equal(nan_a, nan_b) and np.array_equal(a[~nan_a], b[~nan_b]))
    return bool(np.array_equal(a, b))


@functools.lru_cache(maxsize=None)
def config_workload(n: int):
    return wl.WORKLOADS[n]()


@functools.lru_cache(maxsize=None)
def config_oracle(n: int):
    """(k_cache, v_cache, out_fp64, out_bf16) of a named config from the oracle."""
    w = config_workload(n)
    kc, vc = oracle.build_cache(w)
    out, outb = oracle.attend(w, kc, vc)
    return kc, vc, out, outb

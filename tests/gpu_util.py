"""Helpers for the GPU parity tests: move seeded problems to the device, call the
library through its C ABI, and compare with the CPU oracle.

Tolerance (the method's stated bar for floating-point parity): per element
|d - ref| <= 8e-3 * |ref| + 1e-3 * rms(ref), and globally
1 - 2 * sum(d * ref) / sum(d^2 + ref^2) < 1e-3.  Padding rows (+0) and masked
rows (untouched) are compared bit for bit.
"""
import numpy as np
import torch

import moe_grouped_gemm_bf16_gb300 as dg
import workloads as W

REL_TOL = 8e-3
RMS_TOL = 1e-3
GLOBAL_TOL = 1e-3


def bits_to_f64(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(got_bits, ref_bits, what=""):
    g = bits_to_f64(got_bits)
    r = bits_to_f64(ref_bits)
    assert g.shape == r.shape
    if r.size == 0:
        return
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(r * r)))
    err = np.abs(g - r)
    lim = REL_TOL * np.abs(r) + RMS_TOL * rms
    bad = err > lim
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; "
                             f"first {idx.tolist()} got {g[bad][:8]} want {r[bad][:8]}")
    den = float(np.sum(g * g + r * r))
    diff = 1.0 - 2.0 * float(np.sum(g * r)) / den if den > 0 else 0.0
    assert diff < GLOBAL_TOL, f"{what}: global diff {diff}"


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def to_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_dense_add_c(p, C_bits, inplace=False):
    """D = C + A B^T through dg_gemm_fp8_fp8_bf16_nt_add_c; with `inplace` the
    addend buffer is the output."""
    M, N, K = p["M"], p["N"], p["K"]
    A, sa, B, sb = dev(p["A"]), dev(p["sa"]), dev(p["B"]), dev(p["sb"])
    C = dev(np.ascontiguousarray(C_bits).view(np.int16))
    D = C if inplace else torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    dg.gemm_fp8_fp8_bf16_nt_add_c(A, sa, sa.shape[-1], B, sb, C, D, M, N, K)
    torch.cuda.synchronize()
    return to_bits(D)


def run_dense(p, fill=W.BF16_SENTINEL):
    M, N, K = p["M"], p["N"], p["K"]
    A, sa, B, sb = dev(p["A"]), dev(p["sa"]), dev(p["B"]), dev(p["sb"])
    D = torch.full((M, N), 0, dtype=torch.int16, device="cuda")
    D.fill_(np.int16(np.uint16(fill).view(np.int16)))
    dg.gemm_fp8_fp8_bf16_nt(A, sa, sa.shape[-1], B, sb, D, M, N, K)
    torch.cuda.synchronize()
    return to_bits(D)


def run_contiguous(p, fill=W.BF16_SENTINEL):
    M, N, K, G = p["M"], p["N"], p["K"], p["G"]
    A, sa, B, sb = dev(p["A"]), dev(p["sa"]), dev(p["B"]), dev(p["sb"])
    mi = dev(p["m_indices"])
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    D.fill_(np.int16(np.uint16(fill).view(np.int16)))
    dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous(A, sa, sa.shape[-1], B, sb, D, mi, M, N, K, G)
    torch.cuda.synchronize()
    return to_bits(D)


def run_masked(p, expected_m=None, fill=W.BF16_SENTINEL, masked_m=None):
    G, max_m, N, K = p["G"], p["max_m"], p["N"], p["K"]
    A, sa, B, sb = dev(p["A"]), dev(p["sa"]), dev(p["B"]), dev(p["sb"])
    mm = dev(p["masked_m"] if masked_m is None else masked_m)
    D = torch.empty((G, max_m, N), dtype=torch.int16, device="cuda")
    D.fill_(np.int16(np.uint16(fill).view(np.int16)))
    em = expected_m if expected_m is not None else max(1, int(np.mean(p["masked_m"])))
    dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked(A, sa, sa.shape[-1], B, sb, D, mm, G, max_m, N, K,
                                             em)
    torch.cuda.synchronize()
    return to_bits(D)


class forced_config:
    """Context manager: force (block_n, split_k[, pair]) for the launches
    inside (pair: -1 heuristic, 0 off, 1 on).  A configuration the library has
    no kernel for (for example a K split with 256-wide tiles and more than 64
    rows) skips the test."""

    def __init__(self, block_n, split_k, pair=-1):
        self.cfg = (block_n, split_k)
        self.pair = pair

    def __enter__(self):
        dg.debug_force_config(*self.cfg)
        dg.debug_force_pair(self.pair)

    def __exit__(self, exc_type, exc, tb):
        dg.debug_force_config(0, 0)
        dg.debug_force_pair(-1)
        if exc_type is dg.DGError and exc.status == 2 and (self.cfg != (0, 0) or self.pair >= 0):
            import pytest
            pytest.skip(f"no kernel for forced config {self.cfg}")

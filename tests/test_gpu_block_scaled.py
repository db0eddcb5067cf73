"""The block-scaled kernels for packed UE8M0 scales (the tensor cores apply
the scales, tcgen05.mma kind::mxf8f6f4 with block scaling, and accumulate all
of a tile's K in tensor memory) through the C ABI against the CPU oracle:
every instance forced at least once (128-, 224- and 256-wide tiles, the CTA
pair in both widths), in the dense nt, contiguous, masked, nn / tn / tt (with
an addend) and K-grouped forms, on shapes with ragged M and N edges, K group
counts that end inside a packed word, tiles that start inside a 128-column B
block, empty groups and expert padding; then the bench's full-size shapes on
sampled rows."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_bf16_gb300 as dg
import oracle
import workloads as W
from moe_grouped_gemm_bf16_gb300 import _build
from tests import gpu_util as U
from tests.test_gpu_ue8m0 import _sfa, _sfb, dense_ue8m0

pytestmark = pytest.mark.gpu

ORC = None


@pytest.fixture(scope="module", autouse=True)
def built():
    global ORC
    _build.build()
    ORC = oracle.Oracle()
    torch.cuda.init()
    dg.debug_force_block_scaled(1)
    yield
    dg.debug_force_block_scaled(-1)


def _check_status():
    torch.cuda.synchronize()
    assert dg.get_device_status() == 0


def run_dense(p, cfg):
    A, B, sfa, sfb = U.dev(p["A"]), U.dev(p["B"]), U.dev(p["sfa"]), U.dev(p["sfb"])
    D = torch.full((p["M"], p["N"]), -1, dtype=torch.int16, device="cuda")
    with U.forced_config(cfg[0], 0, pair=cfg[1]):
        dg.gemm_fp8_fp8_bf16_nt_ue8m0(A, sfa, sfa.shape[-1], B, sfb, D, p["M"], p["N"], p["K"])
        _check_status()
    return U.to_bits(D)


def test_single_tile_first():
    """One 128 x 128 x 128 tile: the smallest case of the block-scaled MMA."""
    p = dense_ue8m0(128, 128, 128, seed=1)
    got = run_dense(p, (128, 0))
    U.assert_close(got, ORC.gemm_nt_ue8m0(p["A"], p["sfa"], p["B"], p["sfb"]), "single tile")


SHAPES = [(128, 128, 512), (64, 256, 640), (128, 2112, 1152), (200, 400, 2048), (333, 528, 896),
          (1024, 4096, 7168), (520, 7168, 512)]
CFGS = [(0, -1), (128, 0), (224, 0), (256, 0), (128, 1), (256, 1)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: f"bn{c[0]}_p{c[1]}")
def test_dense_block_scaled(shape, cfg):
    M, N, K = shape
    p = dense_ue8m0(M, N, K, seed=M + N + K)
    got = run_dense(p, cfg)
    want = ORC.gemm_nt_ue8m0(p["A"], p["sfa"], p["B"], p["sfb"])
    U.assert_close(got, want, f"block-scaled {shape} cfg={cfg}")


def test_block_scaled_matches_promotion():
    """The block-scaled and the promotion kernels agree (each within the
    tolerance of the oracle; the fp32 sums are ordered differently)."""
    p = dense_ue8m0(384, 1024, 3072, seed=5)
    bs = run_dense(p, (0, -1))
    dg.debug_force_block_scaled(0)
    try:
        pr = run_dense(p, (0, -1))
    finally:
        dg.debug_force_block_scaled(1)
    want = ORC.gemm_nt_ue8m0(p["A"], p["sfa"], p["B"], p["sfb"])
    U.assert_close(bs, want, "block-scaled")
    U.assert_close(pr, want, "promotion")
    U.assert_close(bs, pr, "block-scaled vs promotion")


@pytest.mark.parametrize("bn", [0, 128, 224, 256])
def test_contiguous_block_scaled(bn):
    q = W.contiguous_problem(3, 528, 1152, 100, 300, seed=8 + bn)
    G, K, N = q["G"], q["K"], q["N"]
    kb, ld = K // 128, q["sa"].shape[-1]
    sfa, sfb = _sfa(kb, ld, 9), _sfb((N + 127) // 128, kb, 10, lead=(G,))
    # an all-padding block in the middle (its first row -1)
    mi = q["m_indices"].copy()
    D = torch.full((q["M"], N), -1, dtype=torch.int16, device="cuda")
    with U.forced_config(bn, 0, pair=0):
        dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(
            U.dev(q["A"]), U.dev(sfa), ld, U.dev(q["B"]), U.dev(sfb), D, U.dev(mi), q["M"], N, K, G)
        _check_status()
    want = ORC.grouped_contiguous(q["A"], ORC.decode_sfa(sfa, kb), q["B"],
                                  ORC.decode_sfb(sfb, kb), mi)
    got = U.to_bits(D)
    pad = mi < 0
    assert np.all(got[pad] == 0), "padding rows must be +0"
    U.assert_close(got[~pad], want[~pad], f"contiguous block-scaled bn={bn}")


@pytest.mark.parametrize("cfg", [(0, -1), (128, 0), (256, 0), (128, 1), (256, 1)],
                         ids=lambda c: f"bn{c[0]}_p{c[1]}")
def test_masked_block_scaled(cfg):
    G, max_m, N, K = 6, 384, 528, 1152
    q = W.masked_problem(G, max_m, N, K, 90, seed=12)
    # the edges of the M blocks: empty, one row, a whole block, one past it, full
    mm = np.array([0, 1, 128, 129, 256, 384], np.int32)
    kb, ld = K // 128, q["sa"].shape[-1]
    sfa, sfb = _sfa(kb, ld, 13, lead=(G,)), _sfb((N + 127) // 128, kb, 14, lead=(G,))
    fill = np.uint16(W.BF16_SENTINEL).view(np.int16)
    D = torch.full((G, max_m, N), int(fill), dtype=torch.int16, device="cuda")
    with U.forced_config(cfg[0], 0, pair=cfg[1]):
        dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(
            U.dev(q["A"]), U.dev(sfa), ld, U.dev(q["B"]), U.dev(sfb), D, U.dev(mm), G, max_m, N, K,
            90)
        _check_status()
    init = np.full((G, max_m, N), W.BF16_SENTINEL, np.uint16)
    want = ORC.grouped_masked(q["A"], ORC.decode_sfa(sfa, kb), q["B"], ORC.decode_sfb(sfb, kb),
                              mm, init)
    got = U.to_bits(D)
    for g in range(G):
        v = int(mm[g])
        assert np.array_equal(got[g, v:], want[g, v:]), f"rows past masked_m of group {g}"
        U.assert_close(got[g, :v], want[g, :v], f"masked block-scaled group {g} cfg={cfg}")


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("with_c", [False, True])
def test_layouts_block_scaled(layout, bn, with_c):
    M, N, K = 208, 400, 1152
    p = dense_ue8m0(M, N, K, seed=M + N + K + bn)
    A = np.ascontiguousarray(p["A"].T) if layout[0] == "t" else p["A"]
    B = np.ascontiguousarray(p["B"].T) if layout[1] == "n" else p["B"]
    g = torch.Generator().manual_seed(M + N)
    C = (torch.randn(M, N, generator=g) * 4).to(torch.bfloat16).view(torch.int16)
    D = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    with U.forced_config(bn, 0, pair=0):
        getattr(dg, f"gemm_fp8_fp8_bf16_{layout}_ue8m0")(
            U.dev(A), U.dev(p["sfa"]), p["sfa"].shape[-1], U.dev(B), U.dev(p["sfb"]), D, M, N, K,
            C=C.cuda() if with_c else None)
        _check_status()
    kb = K // 128
    want = ORC.gemm_layout(layout, A, ORC.decode_sfa(p["sfa"], kb), B,
                           ORC.decode_sfb(p["sfb"], kb),
                           C.numpy().view(np.uint16) if with_c else None)
    U.assert_close(U.to_bits(D), want, f"{layout} block-scaled bn={bn} C={with_c}")


@pytest.mark.parametrize("ks", [[256, 0, 384, 640], [1152], [128, 512, 0, 896, 384]],
                         ids=lambda k: "_".join(map(str, k)))
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("with_c", [False, True])
def test_k_grouped_block_scaled(ks, bn, with_c):
    """K-grouped tn: group segments start at any K group, inside a packed
    word; an empty group gives C (or +0)."""
    M, N = 208, 400
    p = W.k_grouped_problem(ks, M, N, seed=sum(ks))
    kb, ld = p["K"] // 128, p["sa"].shape[-1]
    sfa, sfb = _sfa(kb, ld, 21), _sfb((N + 127) // 128, kb, 22)
    G = len(ks)
    g = torch.Generator().manual_seed(G + M)
    C = (torch.randn(G, M, N, generator=g) * 4).to(torch.bfloat16).view(torch.int16)
    D = torch.full((G, M, N), -1, dtype=torch.int16, device="cuda")
    with U.forced_config(bn, 0, pair=0):
        dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0(
            U.dev(p["A"]), U.dev(sfa), ld, U.dev(p["B"]), U.dev(sfb), D, U.dev(p["ks"]), G, M, N,
            p["K"], C=C.cuda() if with_c else None)
        _check_status()
    Cb = C.numpy().view(np.uint16)
    want = ORC.k_grouped_tn(p["A"], ORC.decode_sfa(sfa, kb), p["B"], ORC.decode_sfb(sfb, kb),
                            p["ks"], Cb if with_c else None)
    got = U.to_bits(D)
    for gi in range(G):
        if ks[gi] == 0:
            if with_c:
                assert np.array_equal(got[gi], Cb[gi]), f"empty group {gi} must return C"
            else:
                assert not np.any(got[gi]), f"empty group {gi}"
        else:
            U.assert_close(got[gi], want[gi], f"k-grouped block-scaled {ks} group {gi}")


# ------------------------------------------------ bench shapes, sampled rows --
def _rows(lo, hi, seed):
    rng = np.random.default_rng(seed)
    rows = {lo, hi - 1}
    for b0 in range(lo, hi, 128):
        rows.add(int(rng.integers(b0, min(hi, b0 + 128))))
    return np.array(sorted(rows), np.int64)


@pytest.mark.parametrize("nk", [(7168, 16384), (2112, 7168), (24576, 1536)],
                         ids=lambda s: "x".join(map(str, s)))
def test_prefill_fullsize_block_scaled(nk):
    N, K = nk
    M = 4096
    p = W.dense_problem(M, N, K, seed=W.CONFIGS["dense_prefill"]["seed"])
    sfa, sfb, sa2, sb2 = W.ue8m0_packed_scales(p["sa"], p["sb"])
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.gemm_fp8_fp8_bf16_nt_ue8m0(U.dev(p["A"]), U.dev(sfa), sfa.shape[-1], U.dev(p["B"]),
                                  U.dev(sfb), D, M, N, K)
    _check_status()
    got = U.to_bits(D)
    rows = _rows(0, M, N)
    want = ORC.gemm_nt_rows(p["A"], sa2, p["B"], sb2, rows)
    U.assert_close(got[rows], want, f"prefill block-scaled {nk}")


@pytest.mark.parametrize("nk", W.GROUPED_NK, ids=lambda s: "x".join(map(str, s)))
def test_contiguous_fullsize_block_scaled(nk):
    N, K = nk
    cfg = W.CONFIGS["grouped_contiguous"]
    p = W.contiguous_problem(cfg["groups"], N, K, *cfg["m_range"], seed=cfg["seed"])
    sfa, sfb, sa2, sb2 = W.ue8m0_packed_scales(p["sa"], p["sb"])
    mi = p["m_indices"]
    D = torch.empty((p["M"], N), dtype=torch.int16, device="cuda")
    dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(
        U.dev(p["A"]), U.dev(sfa), sfa.shape[-1], U.dev(p["B"]), U.dev(sfb), D, U.dev(mi), p["M"],
        N, K, p["G"])
    _check_status()
    got = U.to_bits(D)
    assert np.all(got[mi < 0] == 0)
    rows = []
    for e in range(p["G"]):
        r = np.nonzero(mi == e)[0]
        rows += _rows(int(r[0]), int(r[-1]) + 1, e).tolist()
    rows = np.array(sorted(set(rows)), np.int64)
    want = ORC.grouped_contiguous(p["A"], sa2, p["B"], sb2, mi, rows=rows)
    U.assert_close(got[rows], want, f"contiguous block-scaled {nk}")

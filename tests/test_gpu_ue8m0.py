"""Packed UE8M0 scales through the C ABI against the CPU oracle, on the kernels
that decode the scales into the per-K-group promotion (the block-scaled
kernels, which the heuristic prefers for these entry points, are switched off
here and tested in their own module): the dense, contiguous and masked GEMMs
(every dense instance forced, K splits whose slices start inside a packed
word), and the UE8M0 quantiser bit for bit."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_bf16_gb300 as dg
import oracle
import workloads as W
from moe_grouped_gemm_bf16_gb300 import _build
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

ORC = None


@pytest.fixture(scope="module", autouse=True)
def built():
    global ORC
    _build.build()
    ORC = oracle.Oracle()
    torch.cuda.init()
    dg.debug_force_block_scaled(0)
    yield
    dg.debug_force_block_scaled(-1)


def _exponents(shape, seed, lo=118, hi=136):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi, shape, generator=g, dtype=torch.int32).to(torch.uint8).numpy()


def _pack(codes):
    """uint8 [..., n] -> int32 [..., ceil(n/4)], first code in the lowest byte."""
    n = codes.shape[-1]
    pad = (-n) % 4
    if pad:
        codes = np.concatenate([codes, np.zeros(codes.shape[:-1] + (pad,), np.uint8)], axis=-1)
    return np.ascontiguousarray(codes).view("<i4")


def _sfa(kb, ld, seed, lead=()):
    e = _exponents(lead + (ld, kb), seed)                        # [..., ld, kb]
    return np.ascontiguousarray(np.swapaxes(_pack(e), -1, -2))  # [..., ceil(kb/4), ld]


def _sfb(nb, kb, seed, lead=()):
    return _pack(_exponents(lead + (nb, kb), seed))             # [..., nb, ceil(kb/4)]


def dense_ue8m0(M, N, K, seed):
    ld = W.tma_aligned_ld(M)
    return dict(A=W.random_codes((M, K), seed), B=W.random_codes((N, K), seed + 1),
                sfa=_sfa(K // 128, ld, seed + 2), sfb=_sfb((N + 127) // 128, K // 128, seed + 3),
                M=M, N=N, K=K)


def run_dense(p):
    A, B, sfa, sfb = U.dev(p["A"]), U.dev(p["B"]), U.dev(p["sfa"]), U.dev(p["sfb"])
    D = torch.full((p["M"], p["N"]), -1, dtype=torch.int16, device="cuda")
    dg.gemm_fp8_fp8_bf16_nt_ue8m0(A, sfa, sfa.shape[-1], B, sfb, D, p["M"], p["N"], p["K"])
    torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    return U.to_bits(D)


SHAPES = [(64, 256, 640), (128, 2112, 1152), (200, 400, 2048), (333, 528, 896), (1024, 4096, 7168)]
CFGS = [(0, 0, -1), (128, 1, 0), (256, 1, 0), (128, 3, 0), (128, 5, 0), (256, 3, 0), (128, 7, 0),
        (256, 1, 1), (128, 1, 1), (64, 1, 0), (64, 4, 0)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: f"bn{c[0]}_s{c[1]}_p{c[2]}")
def test_dense_ue8m0(shape, cfg):
    M, N, K = shape
    p = dense_ue8m0(M, N, K, seed=M + N + K)
    with U.forced_config(cfg[0], cfg[1], pair=cfg[2]):
        got = run_dense(p)
    want = ORC.gemm_nt_ue8m0(p["A"], p["sfa"], p["B"], p["sfb"])
    U.assert_close(got, want, f"ue8m0 {shape} cfg={cfg}")


@pytest.mark.parametrize("cfg", [(128, 1), (256, 1), (128, 3)], ids=lambda c: f"bn{c[0]}_s{c[1]}")
def test_same_scales_same_bits(cfg):
    """Power-of-two scales given packed or as fp32 give the same bits on the
    same kernel configuration (the two forms' instance tables differ, so the
    heuristic may pick different tilings, whose K-split sums round apart)."""
    M, N, K = 256, 512, 1664
    p = dense_ue8m0(M, N, K, seed=4)
    sa = ORC.decode_sfa(p["sfa"], K // 128)
    sb = ORC.decode_sfb(p["sfb"], K // 128)
    with U.forced_config(*cfg):
        ref = U.run_dense(dict(A=p["A"], sa=sa, B=p["B"], sb=sb, M=M, N=N, K=K))
        got = run_dense(p)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("cfg", [(0, 0), (128, 0), (256, 0)], ids=lambda c: f"bn{c[0]}")
def test_contiguous_ue8m0(cfg):
    q = W.contiguous_problem(3, 400, 1152, 100, 300, seed=8)
    G, K, N = q["G"], q["K"], q["N"]
    kb, ld = K // 128, q["sa"].shape[-1]
    sfa, sfb = _sfa(kb, ld, 9), _sfb((N + 127) // 128, kb, 10, lead=(G,))
    A, B = U.dev(q["A"]), U.dev(q["B"])
    D = torch.full((q["M"], N), -1, dtype=torch.int16, device="cuda")
    with U.forced_config(*cfg):
        dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(A, U.dev(sfa), ld, B, U.dev(sfb), D,
                                                           U.dev(q["m_indices"]), q["M"], N, K, G)
        torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    want = ORC.grouped_contiguous(q["A"], ORC.decode_sfa(sfa, kb), q["B"],
                                  ORC.decode_sfb(sfb, kb), q["m_indices"])
    got = U.to_bits(D)
    pad = q["m_indices"] < 0
    assert np.all(got[pad] == 0)
    U.assert_close(got[~pad], want[~pad], "contiguous ue8m0")


@pytest.mark.parametrize("cfg", [(0, 0), (64, 0), (128, 0), (256, 0)], ids=lambda c: f"bn{c[0]}")
def test_masked_ue8m0(cfg):
    q = W.masked_problem(4, 256, 528, 1152, 90, seed=12)
    G, K, N, max_m = q["G"], q["K"], q["N"], q["max_m"]
    kb, ld = K // 128, q["sa"].shape[-1]
    sfa, sfb = _sfa(kb, ld, 13, lead=(G,)), _sfb((N + 127) // 128, kb, 14, lead=(G,))
    fill = np.uint16(U.W.BF16_SENTINEL).view(np.int16)
    D = torch.full((G, max_m, N), int(fill), dtype=torch.int16, device="cuda")
    with U.forced_config(*cfg, pair=0 if cfg[0] else -1):
        dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(U.dev(q["A"]), U.dev(sfa), ld, U.dev(q["B"]),
                                                       U.dev(sfb), D, U.dev(q["masked_m"]), G,
                                                       max_m, N, K, 90)
        torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    init = np.full((G, max_m, N), U.W.BF16_SENTINEL, np.uint16)
    want = ORC.grouped_masked(q["A"], ORC.decode_sfa(sfa, kb), q["B"], ORC.decode_sfb(sfb, kb),
                              q["masked_m"], init)
    got = U.to_bits(D)
    for g in range(G):
        v = int(q["masked_m"][g])
        assert np.array_equal(got[g, v:], want[g, v:]), f"rows past masked_m of group {g}"
        U.assert_close(got[g, :v], want[g, :v], f"masked ue8m0 group {g}")


def _act(G, M, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(G, M, K, generator=g)
    x *= torch.exp2(torch.randint(-30, 30, (G, M, K // 128), generator=g).float()).repeat_interleave(128, -1)
    if M >= 3:
        x[0, 0, :128] = 0.0
        x[0, 1, :128] = 448.0 * 8.0          # amax exactly 448 * 2^3
        x[0, 2, :128] = 1e-7
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("shape", [(1, 1, 128, 4), (1, 37, 640, 40), (3, 65, 1152, 68),
                                   (1, 4096, 7168, 4096)], ids=lambda s: "x".join(map(str, s)))
def test_quantiser_ue8m0(shape):
    G, M, K, ld = shape
    bits = _act(G, M, K, seed=M + K)
    X = U.dev(bits.view(np.int16))
    Q = torch.empty((G, M, K), dtype=torch.uint8, device="cuda")
    fill = 0x5A5A5A5A
    kbp = (K // 128 + 3) // 4
    sfa = torch.full((G, kbp, ld), fill, dtype=torch.int32, device="cuda")
    dg.quantize_fp8_1x128_ue8m0(X, Q, sfa, G, M, K, ld)
    torch.cuda.synchronize()
    Qr, sfr = ORC.quantize_1x128_ue8m0(bits, ld=ld, fill=fill)
    assert np.array_equal(Q.cpu().numpy(), Qr), "codes differ"
    assert np.array_equal(sfa.cpu().numpy(), sfr), "packed scales differ"


def test_quantiser_then_gemm_ue8m0():
    """GPU UE8M0 quantiser -> GPU UE8M0 GEMM equals the oracle's chain."""
    M, N, K = 200, 384, 1152
    bits = _act(1, M, K, seed=6)[0]
    ld = W.tma_aligned_ld(M)
    Q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(((K // 128 + 3) // 4, ld), dtype=torch.int32, device="cuda")
    dg.quantize_fp8_1x128_ue8m0(U.dev(bits.view(np.int16)), Q, sfa, 1, M, K, ld)
    B = W.random_codes((N, K), 7)
    sfb = _sfb((N + 127) // 128, K // 128, 8)
    D = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.gemm_fp8_fp8_bf16_nt_ue8m0(Q, sfa, ld, U.dev(B), U.dev(sfb), D, M, N, K)
    torch.cuda.synchronize()
    Qr, sfr = ORC.quantize_1x128_ue8m0(bits, ld=ld)
    U.assert_close(U.to_bits(D), ORC.gemm_nt_ue8m0(Qr, sfr, B, sfb), "quantise -> gemm ue8m0")


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
@pytest.mark.parametrize("shape", [(208, 400, 1152), (512, 2112, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("split", [0, 3])
def test_layouts_ue8m0(layout, shape, split):
    """The nn / tn / tt layouts with packed UE8M0 scales (also K-split, whose
    slices start inside a packed word), with an addend."""
    M, N, K = shape
    p = dense_ue8m0(M, N, K, seed=M + N + K + split)
    A = np.ascontiguousarray(p["A"].T) if layout[0] == "t" else p["A"]
    B = np.ascontiguousarray(p["B"].T) if layout[1] == "n" else p["B"]
    g = torch.Generator().manual_seed(M + N)
    C = (torch.randn(M, N, generator=g) * 4).to(torch.bfloat16).view(torch.int16)
    D = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    with U.forced_config(128 if split else 0, split, pair=0 if split else -1):
        getattr(dg, f"gemm_fp8_fp8_bf16_{layout}_ue8m0")(
            U.dev(A), U.dev(p["sfa"]), p["sfa"].shape[-1], U.dev(B), U.dev(p["sfb"]), D, M, N, K,
            C=C.cuda())
        torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    kb = K // 128
    want = ORC.gemm_layout(layout, A, ORC.decode_sfa(p["sfa"], kb), B, ORC.decode_sfb(p["sfb"], kb),
                           C.numpy().view(np.uint16))
    U.assert_close(U.to_bits(D), want, f"{layout} ue8m0 {shape} split={split}")


@pytest.mark.parametrize("ks", [[256, 0, 384, 640], [1152], [128, 512, 0, 896, 384]],
                         ids=lambda k: "_".join(map(str, k)))
def test_k_grouped_ue8m0(ks):
    """K-grouped tn with packed UE8M0 scales: group segments start at any K
    group, so a ring slot's groups can straddle two packed words."""
    M, N = 208, 400
    p = W.k_grouped_problem(ks, M, N, seed=sum(ks))
    kb, ld = p["K"] // 128, p["sa"].shape[-1]
    sfa, sfb = _sfa(kb, ld, 21), _sfb((N + 127) // 128, kb, 22)
    G = len(ks)
    D = torch.full((G, M, N), -1, dtype=torch.int16, device="cuda")
    dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0(
        U.dev(p["A"]), U.dev(sfa), ld, U.dev(p["B"]), U.dev(sfb), D, U.dev(p["ks"]), G, M, N,
        p["K"])
    torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    want = ORC.k_grouped_tn(p["A"], ORC.decode_sfa(sfa, kb), p["B"], ORC.decode_sfb(sfb, kb),
                            p["ks"])
    got = U.to_bits(D)
    for g in range(G):
        if ks[g] == 0:
            assert not np.any(got[g]), f"empty group {g}"
        else:
            U.assert_close(got[g], want[g], f"k-grouped ue8m0 {ks} group {g}")

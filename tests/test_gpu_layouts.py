"""The nn / tn / tt dense layouts and the K-grouped tn form (MN-major operands)
against the CPU oracle, through the C ABI: every instance of each form forced,
ragged M and N, the optional addend C (also in place), K-grouped groups
without K rows, and a bad ks entry reported by the device status word."""
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


def _addend(shape, seed):
    g = torch.Generator().manual_seed(seed)
    c = torch.randn(*shape, generator=g) * 4.0
    return c.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _stored(p, layout):
    """The dense problem's operands in the storage `layout` names."""
    A = np.ascontiguousarray(p["A"].T) if layout[0] == "t" else p["A"]
    B = np.ascontiguousarray(p["B"].T) if layout[1] == "n" else p["B"]
    return A, B


def run_layout(layout, p, C=None, inplace=False):
    M, N, K = p["M"], p["N"], p["K"]
    A, B = _stored(p, layout)
    A, B, sa, sb = U.dev(A), U.dev(B), U.dev(p["sa"]), U.dev(p["sb"])
    Cd = U.dev(np.ascontiguousarray(C).view(np.int16)) if C is not None else None
    D = Cd if inplace else torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    getattr(dg, "gemm_fp8_fp8_bf16_" + layout)(A, sa, sa.shape[-1], B, sb, D, M, N, K, C=Cd)
    torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    return U.to_bits(D)


LAYOUTS = ["nn", "tn", "tt"]
SHAPES = [(64, 144, 640), (208, 400, 384), (336, 2112, 256), (512, 528, 1024), (1024, 4096, 2048)]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("bn", [0, 128, 256])
def test_dense_layout(layout, shape, bn):
    M, N, K = shape
    p = W.dense_problem(M, N, K, seed=M + 3 * N + K)
    with U.forced_config(bn, 0, pair=-1):
        got = run_layout(layout, p)
    A, B = _stored(p, layout)
    U.assert_close(got, ORC.gemm_layout(layout, A, p["sa"], B, p["sb"]), f"{layout} {shape} bn={bn}")


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("inplace", [False, True])
def test_dense_layout_add_c(layout, inplace):
    M, N, K = 208, 400, 512
    p = W.dense_problem(M, N, K, seed=91)
    C = _addend((M, N), seed=92)
    got = run_layout(layout, p, C, inplace=inplace)
    A, B = _stored(p, layout)
    U.assert_close(got, ORC.gemm_layout(layout, A, p["sa"], B, p["sb"], C), f"{layout} add_c")


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", [(64, 2112, 1024), (128, 4096, 2048), (208, 400, 384)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("split", [2, 3, 5])
@pytest.mark.parametrize("with_c", [False, True])
def test_dense_layout_split(layout, shape, split, with_c):
    """The K split over a cluster with MN-major operands (the decode shapes'
    configuration), with and without the addend."""
    M, N, K = shape
    p = W.dense_problem(M, N, K, seed=M + N + K + split)
    C = _addend((M, N), seed=M + split) if with_c else None
    with U.forced_config(128, split, pair=0):
        got = run_layout(layout, p, C)
    A, B = _stored(p, layout)
    U.assert_close(got, ORC.gemm_layout(layout, A, p["sa"], B, p["sb"], C),
                   f"{layout} {shape} split={split} C={with_c}")


def test_layouts_agree_with_nt():
    """All four storages of one logical problem give the same bits (same
    arithmetic, only the operands' shared-memory layout differs)."""
    p = W.dense_problem(256, 512, 1024, seed=5)
    for bn in (128, 256):
        with U.forced_config(bn, 1, pair=0):   # the same tiles, no K split
            ref = U.run_dense(p)
            for layout in LAYOUTS:
                assert np.array_equal(run_layout(layout, p), ref), f"{layout} bn={bn}"


def _spare_rows(p):
    """Operands with 128 extra K rows that no group owns (sum(ks) < K_total
    is allowed): random codes and scales, which must not reach D."""
    M, N = p["M"], p["N"]
    A = np.concatenate([p["A"], W.random_codes((128, M), seed=1)])
    B = np.concatenate([p["B"], W.random_codes((128, N), seed=2)])
    sa = np.concatenate([p["sa"], np.ones((1, p["sa"].shape[1]), np.float32)])
    sb = np.concatenate([p["sb"], np.ones((p["sb"].shape[0], 1), np.float32)], axis=1)
    return A, B, sa, sb, p["K"] + 128


def run_k_grouped(p, C=None, inplace=False, ks_dev=None, spare=False):
    M, N, K, G = p["M"], p["N"], p["K"], p["G"]
    A, B, sa, sb = p["A"], p["B"], p["sa"], p["sb"]
    if spare:
        A, B, sa, sb, K = _spare_rows(p)
    A, B, sa, sb = U.dev(A), U.dev(B), U.dev(sa), U.dev(sb)
    ks = U.dev(p["ks"] if ks_dev is None else ks_dev)
    Cd = U.dev(np.ascontiguousarray(C).view(np.int16)) if C is not None else None
    D = Cd if inplace else torch.full((G, M, N), -1, dtype=torch.int16, device="cuda")
    dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(A, sa, sa.shape[-1], B, sb, D, ks, G, M, N, K,
                                                 C=Cd)
    torch.cuda.synchronize()
    return U.to_bits(D)


KS_CASES = [
    ([512], 128, 256),
    ([256, 0, 384, 128, 640], 208, 400),
    ([128] * 9, 336, 272),
    ([1024, 2048, 0], 512, 2112),
    ([0, 0], 128, 256),
]


@pytest.mark.parametrize("case", KS_CASES, ids=lambda c: f"G{len(c[0])}_M{c[1]}_N{c[2]}")
@pytest.mark.parametrize("bn", [0, 128, 256])
@pytest.mark.parametrize("with_c", [False, True])
def test_k_grouped(case, bn, with_c):
    ks, M, N = case
    p = W.k_grouped_problem(ks, M, N, seed=sum(ks) + M + N)
    C = _addend((len(ks), M, N), seed=M * N) if with_c else None
    with U.forced_config(bn, 0, pair=-1):
        # all groups empty: K_total must still be >= 128, so pass 128 unowned rows
        got = run_k_grouped(p, C, spare=p["K"] == 0)
    assert dg.get_device_status() == 0
    want = ORC.k_grouped_tn(p["A"], p["sa"], p["B"], p["sb"], p["ks"], C)
    for g in range(len(ks)):
        if ks[g] == 0:   # no K rows: D = C or +0, bit for bit
            assert np.array_equal(got[g], want[g]), f"empty group {g}"
        else:
            U.assert_close(got[g], want[g], f"k-grouped {case} bn={bn} group {g}")


def test_k_grouped_in_place():
    ks, M, N = [384, 256, 0, 512], 256, 512
    p = W.k_grouped_problem(ks, M, N, seed=7)
    C = _addend((len(ks), M, N), seed=8)
    got = run_k_grouped(p, C, inplace=True)
    U.assert_close(got, ORC.k_grouped_tn(p["A"], p["sa"], p["B"], p["sb"], p["ks"], C), "in place")


def test_k_grouped_wgrad_shape():
    """One expert group set at the bench's weight-gradient shape, checked on
    sampled rows of every group (the oracle computes the sampled rows only,
    by slicing each group's K range)."""
    ks = W.random_ks(4, 2048, 6144, seed=3)
    M, N = 4096, 7168
    p = W.k_grouped_problem(ks, M, N, seed=11)
    got = run_k_grouped(p)
    rows = np.array([0, 1, 127, 128, 2047, 4000, 4095])
    k0 = 0
    for g, kg in enumerate(ks):
        j0, j1 = k0 // 128, (k0 + kg) // 128
        Ag = np.ascontiguousarray(p["A"][k0:k0 + kg, rows].T)
        Bg = np.ascontiguousarray(p["B"][k0:k0 + kg].T)
        sag = np.ascontiguousarray(p["sa"][j0:j1][:, rows])
        sbg = np.ascontiguousarray(p["sb"][:, j0:j1])
        want = ORC.gemm_nt(Ag, sag, Bg, sbg)
        U.assert_close(got[g][rows], want, f"wgrad group {g}")
        k0 += kg


def test_k_grouped_unowned_rows_ignored():
    """K rows past sum(ks) belong to no group and do not reach D."""
    ks, M, N = [256, 384], 208, 400
    p = W.k_grouped_problem(ks, M, N, seed=17)
    got = run_k_grouped(p, spare=True)
    assert dg.get_device_status() == 0
    want = ORC.k_grouped_tn(p["A"], p["sa"], p["B"], p["sb"], p["ks"])
    for g in range(len(ks)):
        U.assert_close(got[g], want[g], f"group {g}")


def test_k_grouped_bad_ks_reported():
    """A ks entry that is not whole K groups is clamped and reported."""
    ks, M, N = [256, 384], 128, 256
    p = W.k_grouped_problem(ks, M, N, seed=13)
    bad = np.array([256, 200], np.int32)   # 200 is not a multiple of 128
    run_k_grouped(p, ks_dev=bad)
    assert dg.get_device_status() == 10
    assert dg.get_device_status() == 0


def test_k_grouped_graph_follows_device_ks():
    """One captured launch; the group sizes change on the device between
    replays (the host never reads ks), and each replay computes the new split
    of the same K rows."""
    ks1, ks2 = [256, 384, 128], [640, 0, 128]          # both sum to 768
    M, N = 208, 400
    p = W.k_grouped_problem(ks1, M, N, seed=31)
    A, B, sa, sb = U.dev(p["A"]), U.dev(p["B"]), U.dev(p["sa"]), U.dev(p["sb"])
    ks = U.dev(np.asarray(ks1, np.int32))
    D = torch.zeros((3, M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    call = lambda: dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(
        A, sa, sa.shape[-1], B, sb, D, ks, 3, M, N, p["K"], stream=s.cuda_stream)
    with torch.cuda.stream(s):
        call()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call()
    for kk in (ks1, ks2):
        ks.copy_(torch.from_numpy(np.asarray(kk, np.int32)))
        g.replay()
        torch.cuda.synchronize()
        want = ORC.k_grouped_tn(p["A"], p["sa"], p["B"], p["sb"], np.asarray(kk, np.int32))
        got = U.to_bits(D)
        for gi in range(3):
            if kk[gi] == 0:
                assert not np.any(got[gi]), f"ks={kk}: empty group {gi}"
            else:
                U.assert_close(got[gi], want[gi], f"graph ks={kk} group {gi}")
    assert dg.get_device_status() == 0

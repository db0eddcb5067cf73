"""Degenerate and extreme inputs of the grouped forms, through the C ABI,
against the CPU oracle: every masked group empty, every contiguous block
padding, the smallest shapes, and the largest group count the masked form
takes (1024)."""
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
    yield
    dg.debug_force_config(0, 0)
    dg.debug_force_pair(-1)


def _check_masked(p, mm, what):
    got = U.run_masked(p, masked_m=mm, expected_m=max(1, int(mm.mean())))
    assert dg.get_device_status() == 0, what
    init = np.full(got.shape, W.BF16_SENTINEL, np.uint16)
    want = ORC.grouped_masked(p["A"], p["sa"], p["B"], p["sb"], mm, init)
    for g in range(p["G"]):
        v = int(mm[g])
        assert np.all(got[g, v:] == W.BF16_SENTINEL), f"{what}: group {g} rows past masked_m written"
        U.assert_close(got[g, :v], want[g, :v], f"{what}: group {g}")


@pytest.mark.parametrize("cfg", [(0, 0, -1), (128, 1, 0), (256, 1, 1)],
                         ids=lambda c: f"bn{c[0]}_pair{c[2]}")
def test_masked_all_groups_empty(cfg):
    """No group has a row: no tile exists, D is left as it was."""
    p = W.masked_problem(4, 256, 528, 1024, 64, seed=301)
    mm = np.zeros(4, np.int32)
    dg.get_device_status()
    with U.forced_config(*cfg):
        _check_masked(p, mm, f"all empty {cfg}")


def test_contiguous_all_padding():
    """Every 128-row block is padding (m_indices = -1): D is all +0."""
    p = W.contiguous_problem(2, 272, 512, 1, 100, seed=303)
    p = dict(p)
    p["m_indices"] = np.full(p["M"], -1, np.int32)
    dg.get_device_status()
    got = U.run_contiguous(p)
    assert dg.get_device_status() == 0
    assert np.all(got == 0)


def test_smallest_shapes():
    """One K group, N = 16, one row: masked (G = 1, max_m = 1) and
    contiguous (one expert of one valid row in a 128-row block)."""
    p = W.masked_problem(1, 1, 16, 128, 1, seed=305)
    _check_masked(p, np.array([1], np.int32), "masked 1x16x128")
    q = W.contiguous_problem(1, 16, 128, 1, 1, seed=307)
    got = U.run_contiguous(q)
    assert dg.get_device_status() == 0
    want = ORC.grouped_contiguous(q["A"], q["sa"], q["B"], q["sb"], q["m_indices"])
    pad = q["m_indices"] < 0
    assert np.all(got[pad] == 0)
    U.assert_close(got[~pad], want[~pad], "contiguous 1 row")


def test_masked_most_groups():
    """1024 groups (the largest count), each with 0..16 rows: the device's
    prefix of M blocks spans 32 warp passes."""
    p = W.masked_problem(1024, 16, 32, 128, 8, seed=309, m_lo=0)
    mm = p["masked_m"].copy()
    assert (mm == 0).any() and (mm == 16).any()
    dg.get_device_status()
    _check_masked(p, mm, "1024 groups")


def test_b_scales_not_16_byte_aligned():
    """sb only 4-byte aligned (allowed by the ABI): the producer's bulk copy of
    a tile's B-scale rows then starts up to 12 bytes before the first row (the
    16-byte boundary below it) and the promotion reads from that offset.
    Dense and masked, against the oracle."""
    p = W.dense_problem(200, 400, 1024, seed=311)
    M, N, K = p["M"], p["N"], p["K"]
    A, sa, B = U.dev(p["A"]), U.dev(p["sa"]), U.dev(p["B"])
    sb_flat = np.concatenate([np.zeros(1, np.float32), p["sb"].ravel()])
    sb_buf = U.dev(sb_flat)
    sb = sb_buf[1:]                      # 4 bytes past a 16-byte boundary
    assert sb.data_ptr() % 16 == 4
    D = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    dg.get_device_status()
    dg.gemm_fp8_fp8_bf16_nt(A, sa, sa.shape[-1], B, sb, D, M, N, K)
    torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    U.assert_close(U.to_bits(D), ORC.gemm_nt(p["A"], p["sa"], p["B"], p["sb"]), "dense, sb + 4 B")

    q = W.masked_problem(3, 256, 400, 1024, 90, seed=313)
    mm = q["masked_m"].copy()
    A, sa, B = U.dev(q["A"]), U.dev(q["sa"]), U.dev(q["B"])
    sb_buf = U.dev(np.concatenate([np.zeros(1, np.float32), q["sb"].ravel()]))
    sb = sb_buf[1:]
    D = torch.full((3, 256, 400), -1, dtype=torch.int16, device="cuda")
    dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked(A, sa, sa.shape[-1], B, sb, D, U.dev(mm), 3, 256,
                                             400, 1024, 90)
    torch.cuda.synchronize()
    assert dg.get_device_status() == 0
    got = U.to_bits(D)
    init = np.full(got.shape, 0xFFFF, np.uint16)
    want = ORC.grouped_masked(q["A"], q["sa"], q["B"], q["sb"], mm, init)
    for g in range(3):
        v = int(mm[g])
        assert np.all(got[g, v:] == 0xFFFF)
        U.assert_close(got[g, :v], want[g, :v], f"masked, sb + 4 B, group {g}")


@pytest.mark.parametrize("K", [640, 1152, 2560], ids=lambda k: f"K{k}")
def test_packed_b_scales_not_16_byte_aligned(K):
    """Packed UE8M0 B scales (K/512 words per row, rounded up) 4 bytes past a
    16-byte boundary, through the promotion kernels' packed-scale twins (the
    block-scaled kernels switched off): rows of 2, 3 and 5 words, so the tiles'
    spans start at every offset within a 16-byte unit.  Dense and masked."""
    kb, kbp = K // 128, (K // 128 + 3) // 4
    p = W.dense_problem(200, 656, K, seed=315 + K)
    M, N = p["M"], p["N"]
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(K)
    e_a = torch.randint(120, 134, (M, kb), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    e_b = torch.randint(120, 134, (nb, kb), generator=g, dtype=torch.int32).to(torch.uint8).numpy()

    def pack(e):
        pad = (-e.shape[-1]) % 4
        e = np.concatenate([e, np.zeros(e.shape[:-1] + (pad,), np.uint8)], axis=-1)
        return np.ascontiguousarray(e).view("<i4")

    ld = W.tma_aligned_ld(M)
    sfa = np.zeros((kbp, ld), np.int32)
    sfa[:, :M] = pack(e_a).T
    sfb = pack(e_b)                                   # [nb, kbp]
    sb_buf = U.dev(np.concatenate([np.zeros(1, np.int32), sfb.ravel()]))
    sb = sb_buf[1:]
    assert sb.data_ptr() % 16 == 4
    A, B = U.dev(p["A"]), U.dev(p["B"])
    D = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    dg.debug_force_block_scaled(0)
    try:
        dg.get_device_status()
        dg.gemm_fp8_fp8_bf16_nt_ue8m0(A, U.dev(sfa), ld, B, sb, D, M, N, K)
        torch.cuda.synchronize()
        assert dg.get_device_status() == 0
        want = ORC.gemm_nt(p["A"], ORC.decode_sfa(sfa, kb), p["B"], ORC.decode_sfb(sfb, kb))
        U.assert_close(U.to_bits(D), want[:M], f"dense ue8m0, sb + 4 B, K={K}")

        q = W.masked_problem(3, 256, 400, K, 90, seed=317 + K)
        G, mm = 3, q["masked_m"].copy()
        nbq = (400 + 127) // 128
        e_bq = torch.randint(120, 134, (G, nbq, kb), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
        e_aq = torch.randint(120, 134, (G, 256, kb), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
        ldq = q["sa"].shape[-1]
        sfaq = np.zeros((G, kbp, ldq), np.int32)
        sfaq[:, :, :256] = np.swapaxes(pack(e_aq), -1, -2)
        sfbq = pack(e_bq)                             # [G, nbq, kbp]
        sbq = U.dev(np.concatenate([np.zeros(1, np.int32), sfbq.ravel()]))[1:]
        D = torch.full((G, 256, 400), -1, dtype=torch.int16, device="cuda")
        dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(U.dev(q["A"]), U.dev(sfaq), ldq, U.dev(q["B"]),
                                                       sbq, D, U.dev(mm), G, 256, 400, K, 90)
        torch.cuda.synchronize()
        assert dg.get_device_status() == 0
        got = U.to_bits(D)
        init = np.full(got.shape, 0xFFFF, np.uint16)
        want = ORC.grouped_masked(q["A"], ORC.decode_sfa(sfaq, kb), q["B"], ORC.decode_sfb(sfbq, kb),
                                  mm, init)
        for z in range(G):
            v = int(mm[z])
            assert np.all(got[z, v:] == 0xFFFF)
            U.assert_close(got[z, :v], want[z, :v], f"masked ue8m0, sb + 4 B, K={K}, group {z}")
    finally:
        dg.debug_force_block_scaled(-1)

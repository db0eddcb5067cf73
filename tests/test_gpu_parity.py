"""CUDA path vs the CPU oracle, element by element, on seeded inputs small
enough for the oracle to finish in seconds, spanning several tiles and ragged
tails, through the C ABI.  Every kernel instance is exercised by forcing its
configuration, besides the heuristic's own choice."""
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


def dense_ref(p):
    return ORC.gemm_nt(p["A"], p["sa"], p["B"], p["sb"])


# (block_n, split_k): every dense instance, plus the heuristic (0, 0)
DENSE_CONFIGS = [(0, 0), (64, 1), (128, 1), (256, 1), (64, 3), (128, 2), (128, 3), (128, 4),
                 (128, 8), (256, 2), (256, 5), (256, 8)]


@pytest.mark.parametrize("cfg", DENSE_CONFIGS, ids=lambda c: f"bn{c[0]}_s{c[1]}")
def test_dense_tiny_config(cfg):
    """The small dense case: M=128, N=256, K=512."""
    p = W.dense_problem(128, 256, 512, seed=1000)
    with U.forced_config(*cfg):
        got = U.run_dense(p)
    U.assert_close(got, dense_ref(p), f"dense 128x256x512 cfg={cfg}")


RAGGED = [
    (1, 16, 128),        # one row, one column block, one K group
    (64, 144, 640),      # decode-sized M, ragged N tail, 5 K groups
    (200, 400, 384),     # ragged M and N
    (333, 2112, 256),    # the 2112 width: last B scale block is 64 rows
    (512, 528, 1024),    # several M and N tiles
    (130, 272, 128 * 9),  # K groups not divisible by the split
]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("cfg", [(0, 0), (64, 1), (128, 1), (256, 1), (64, 4), (128, 3),
                                 (256, 3)],
                         ids=lambda c: f"bn{c[0]}_s{c[1]}")
def test_dense_ragged(shape, cfg):
    M, N, K = shape
    p = W.dense_problem(M, N, K, seed=M * 7 + N + K)
    with U.forced_config(*cfg):
        got = U.run_dense(p)
    U.assert_close(got, dense_ref(p), f"dense {shape} cfg={cfg}")


def test_dense_more_splits_than_groups():
    """split_k = 8 with only 2 K groups: six CTAs of each cluster get no K
    group and add zeros."""
    p = W.dense_problem(96, 256, 256, seed=5)
    with U.forced_config(128, 8):
        got = U.run_dense(p)
    U.assert_close(got, dense_ref(p), "split 8 > K groups")


def test_dense_special_values():
    """Integer-valued codes and power-of-two scales: the exact answer is an
    integer, which bf16 holds exactly below 256 (sparse inputs)."""
    rng = np.random.default_rng(3)
    M, N, K = 256, 384, 512
    A = np.where(rng.random((M, K)) < 0.02, 0x38, 0).astype(np.uint8)  # 1.0 or 0
    B = np.where(rng.random((N, K)) < 0.05, 0xC0, 0).astype(np.uint8)  # -2.0 or 0
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones(((N + 127) // 128, K // 128), np.float32)
    p = dict(A=A, sa=sa, B=B, sb=sb, M=M, N=N, K=K)
    got = U.run_dense(p)
    want = dense_ref(p)
    assert np.array_equal(got, want)


def test_dense_repeat_is_deterministic():
    p = W.dense_problem(64, 2112, 1024, seed=9)
    a = U.run_dense(p)
    b = U.run_dense(p)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("cfg", [(0, 0), (128, 1), (256, 1)], ids=lambda c: f"bn{c[0]}")
def test_contiguous_small(cfg):
    p = W.contiguous_problem(3, 272, 384, 1, 300, seed=31)
    with U.forced_config(*cfg):
        got = U.run_contiguous(p)
    want = ORC.grouped_contiguous(p["A"], p["sa"], p["B"], p["sb"], p["m_indices"])
    pad = p["m_indices"] < 0
    assert pad.any()
    assert np.all(got[pad] == 0), "padding rows must be +0"
    U.assert_close(got[~pad], want[~pad], f"contiguous cfg={cfg}")


def test_contiguous_all_padding_block():
    """A 128-row block whose first row is -1 is all padding."""
    p = W.contiguous_problem(2, 128, 256, 5, 100, seed=33)
    M = p["M"]
    # append a whole padding block
    p = dict(p)
    p["A"] = np.concatenate([p["A"], W.random_codes((128, p["K"]), 1)])
    sa = np.ones((p["K"] // 128, W.tma_aligned_ld(M + 128)), np.float32)
    sa[:, :M] = p["sa"][:, :M]
    p["sa"] = sa
    p["m_indices"] = np.concatenate([p["m_indices"], np.full(128, -1, np.int32)])
    p["M"] = M + 128
    got = U.run_contiguous(p)
    want = ORC.grouped_contiguous(p["A"], p["sa"], p["B"], p["sb"], p["m_indices"])
    assert np.all(got[M:] == 0)
    pad = p["m_indices"] < 0
    U.assert_close(got[~pad], want[~pad], "contiguous with padding block")


@pytest.mark.parametrize("cfg", [(0, 0), (128, 1), (256, 1)], ids=lambda c: f"bn{c[0]}")
def test_masked_small(cfg):
    p = W.masked_problem(5, 300, 400, 384, 100, seed=41)
    # edge counts: an empty group, exactly one tile, the full max_m
    mm = p["masked_m"].copy()
    mm[0], mm[1], mm[2] = 0, 128, 300
    p["masked_m"] = mm
    with U.forced_config(*cfg):
        got = U.run_masked(p)
    init = np.full(got.shape, W.BF16_SENTINEL, np.uint16)
    want = ORC.grouped_masked(p["A"], p["sa"], p["B"], p["sb"], mm, init)
    for g in range(p["G"]):
        v = int(mm[g])
        assert np.all(got[g, v:] == W.BF16_SENTINEL), f"group {g}: rows past masked_m written"
        U.assert_close(got[g, :v], want[g, :v], f"masked group {g}")


MASKED_PAIR_CASES = [
    # (G, max_m, N, K, masked_m override)
    (5, 300, 400, 384, [0, 128, 300, 129, 256]),   # empty, one CTA, full, 1 row in the 2nd
    (4, 200, 528, 1024, [200, 57, 1, 128]),         # max_m not a multiple of 256
    (3, 1024, 4096, 2048, [512, 1000, 300]),        # several pair blocks per group
    (8, 512, 4096, 512, [512] * 8),                 # 256-512 pair tiles: several per pair
]


@pytest.mark.parametrize("case", MASKED_PAIR_CASES, ids=lambda c: f"G{c[0]}_m{c[1]}_N{c[2]}_K{c[3]}")
@pytest.mark.parametrize("bn", [128, 256])
def test_masked_pair(case, bn):
    """The masked form over CTA pairs (256-row blocks, each CTA storing only
    its own valid rows; rows past masked_m untouched, bit for bit)."""
    G, max_m, N, K, mm = case
    p = W.masked_problem(G, max_m, N, K, 100, seed=G * 7 + N)
    p["masked_m"] = np.asarray(mm, np.int32)
    with U.forced_config(bn, 1, pair=1):
        got = U.run_masked(p)
    assert dg.get_device_status() == 0
    init = np.full(got.shape, W.BF16_SENTINEL, np.uint16)
    want = ORC.grouped_masked(p["A"], p["sa"], p["B"], p["sb"], p["masked_m"], init)
    for g in range(G):
        v = int(mm[g])
        assert np.all(got[g, v:] == W.BF16_SENTINEL), f"group {g}: rows past masked_m written"
        U.assert_close(got[g, :v], want[g, :v], f"masked pair group {g} bn={bn}")


PAIR_SHAPES = [
    (64, 256, 512),       # the second CTA of the pair has no rows
    (1, 16, 128),
    (200, 400, 384),      # ragged M and N
    (333, 2112, 256),     # 2112: last B scale block is 64 rows
    (512, 528, 1024),
    (2048, 4096, 256),    # 8 x 16 = 128 pair tiles: more than the resident pairs
]


@pytest.mark.parametrize("shape", PAIR_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("bn", [256, 128], ids=lambda b: f"bn{b}")
def test_dense_pair(shape, bn):
    """The CTA-pair form (cta_group::2 MMA over a 2-CTA cluster, 256-row tiles)."""
    M, N, K = shape
    p = W.dense_problem(M, N, K, seed=M * 3 + N * 5 + K)
    with U.forced_config(bn, 1, pair=1):
        got = U.run_dense(p)
    U.assert_close(got, dense_ref(p), f"dense pair {shape}")


def test_dense_pair_off_matches():
    """Pair form forced off on a shape the heuristic gives to the pair form."""
    p = W.dense_problem(640, 768, 512, seed=77)
    with U.forced_config(0, 0, pair=0):
        a = U.run_dense(p)
    with U.forced_config(0, 0, pair=1):
        b = U.run_dense(p)
    want = dense_ref(p)
    U.assert_close(a, want, "pair off")
    U.assert_close(b, want, "pair on")


def test_dense_largest_k():
    """K = 128 * 512, the largest the kernels take (the B-scale staging holds
    three 128-column blocks for every K group)."""
    p = W.dense_problem(64, 272, 128 * 512, seed=31)
    got = U.run_dense(p)
    U.assert_close(got, dense_ref(p), "K = 65536")


def test_graph_replay_sees_new_inputs():
    """The calls capture into a CUDA graph (no host synchronisation, no host
    read of device data); replaying the graph after overwriting the inputs in
    place computes on the new values."""
    p1 = W.dense_problem(200, 384, 1024, seed=41)
    p2 = W.dense_problem(200, 384, 1024, seed=42)
    M, N, K = 200, 384, 1024
    A, sa, B, sb = U.dev(p1["A"]), U.dev(p1["sa"]), U.dev(p1["B"]), U.dev(p1["sb"])
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dg.gemm_fp8_fp8_bf16_nt(A, sa, sa.shape[-1], B, sb, D, M, N, K, s.cuda_stream)  # warm-up
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dg.gemm_fp8_fp8_bf16_nt(A, sa, sa.shape[-1], B, sb, D, M, N, K, s.cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    U.assert_close(U.to_bits(D), dense_ref(p1), "graph replay 1")
    for dst, src in ((A, p2["A"]), (sa, p2["sa"]), (B, p2["B"]), (sb, p2["sb"])):
        dst.copy_(torch.from_numpy(np.ascontiguousarray(src)))
    g.replay()
    torch.cuda.synchronize()
    U.assert_close(U.to_bits(D), dense_ref(p2), "graph replay 2")
    assert dg.get_device_status() == 0


ADD_C_SHAPES = [(64, 144, 640), (200, 400, 384), (333, 2112, 256), (512, 528, 1024)]
ADD_C_CFGS = [(0, 0, -1), (128, 1, 0), (256, 1, 0), (128, 3, 0), (256, 5, 0), (256, 1, 1),
              (128, 1, 1)]


def _addend(M, N, seed):
    g = torch.Generator().manual_seed(seed)
    c = torch.randn(M, N, generator=g) * 4.0
    return c.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("shape", ADD_C_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("cfg", ADD_C_CFGS, ids=lambda c: f"bn{c[0]}_s{c[1]}_p{c[2]}")
def test_dense_add_c(shape, cfg):
    """D = C + A B^T in every dense form (plain, K split with full and 64-row
    A, CTA pair) against the oracle's addend form."""
    M, N, K = shape
    p = W.dense_problem(M, N, K, seed=M + 2 * N + K)
    C = _addend(M, N, seed=M * N)
    with U.forced_config(cfg[0], cfg[1], pair=cfg[2]):
        got = U.run_dense_add_c(p, C)
    want = ORC.gemm_nt_c(p["A"], p["sa"], p["B"], p["sb"], C)
    U.assert_close(got, want, f"add_c {shape} cfg={cfg}")


@pytest.mark.parametrize("cfg", [(0, 0, -1), (128, 3, 0), (256, 1, 1)],
                         ids=lambda c: f"bn{c[0]}_s{c[1]}_p{c[2]}")
def test_dense_add_c_in_place(cfg):
    """C is D: the output buffer accumulates."""
    M, N, K = 130, 272, 512
    p = W.dense_problem(M, N, K, seed=88)
    C = _addend(M, N, seed=89)
    with U.forced_config(cfg[0], cfg[1], pair=cfg[2]):
        got = U.run_dense_add_c(p, C, inplace=True)
    U.assert_close(got, ORC.gemm_nt_c(p["A"], p["sa"], p["B"], p["sb"], C), f"in place {cfg}")


@pytest.mark.parametrize("bn", [128, 256])
def test_contiguous_padding_tiles_last_on_few_sms(bn):
    """A whole padding block at the end, on 3 CTAs: each CTA's last tiles are
    padding tiles, which reuse a B-scale buffer with a plain barrier arrival
    after its last real fill; the CTA's final drain must still see every
    phase complete (no timeout in the status word)."""
    p = W.contiguous_problem(3, 272, 512, 1, 300, seed=231)
    M = p["M"]
    p = dict(p)
    p["A"] = np.concatenate([p["A"], W.random_codes((256, p["K"]), 5)])
    sa = np.ones((p["K"] // 128, W.tma_aligned_ld(M + 256)), np.float32)
    sa[:, :M] = p["sa"][:, :M]
    p["sa"] = sa
    p["m_indices"] = np.concatenate([p["m_indices"], np.full(256, -1, np.int32)])
    p["M"] = M + 256
    dg.get_device_status()   # read and clear
    dg.set_num_sms(3)
    try:
        with U.forced_config(bn, 1):
            got = U.run_contiguous(p)
    finally:
        dg.set_num_sms(0)
    assert dg.get_device_status() == 0
    want = ORC.grouped_contiguous(p["A"], p["sa"], p["B"], p["sb"], p["m_indices"])
    pad = p["m_indices"] < 0
    assert np.all(got[pad] == 0)
    U.assert_close(got[~pad], want[~pad], f"contiguous padding last bn={bn}")

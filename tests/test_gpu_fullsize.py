"""Full-size workloads (the DeepSeek-V3/R1 inference shapes of the pages'
benchmarks), in the configuration the library picks and the bench times.

The GPU computes every output; the oracle recomputes a sample of whole rows
(so every N tile, the last one included, is checked on each sampled row),
compared element by element with the tolerance: at least one seeded row of
every 128-row M block (so every raster band, every M block of every expert and
of every group, and every wave of tiles is touched), plus each M block's first
and last rows where the oracle cost allows.  Properties that hold at any size
are checked on every row: contiguous padding rows are +0 and masked rows past
masked_m keep the sentinel, bit for bit, and no output is non-finite."""
import numpy as np
import pytest
import torch

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


def sample_rows(M, k, seed):
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    rows.update(rng.integers(0, M, size=max(0, k - 2)).tolist())
    return np.array(sorted(rows), np.int64)


def rows_per_block(lo, hi, seed, block=128):
    """One seeded row in every `block`-row block of [lo, hi), plus lo and
    hi - 1."""
    rng = np.random.default_rng(seed)
    rows = {lo, hi - 1}
    for b0 in range(lo, hi, block):
        rows.add(int(rng.integers(b0, min(hi, b0 + block))))
    return sorted(rows)


DECODE = [(m, n, k) for m in (64, 128) for (n, k) in W.DENSE_NK]
PREFILL = [(4096, n, k) for (n, k) in W.DENSE_NK]


@pytest.mark.parametrize("shape", DECODE + PREFILL, ids=lambda s: "x".join(map(str, s)))
def test_dense_fullsize(shape):
    M, N, K = shape
    seed = W.CONFIGS["dense_decode" if M <= 128 else "dense_prefill"]["seed"]
    p = W.dense_problem(M, N, K, seed=seed)
    got = U.run_dense(p)
    assert np.all(np.isfinite(U.bits_to_f64(got)))
    if M <= 128:
        rows = sample_rows(M, 16, seed + N)
    else:
        # every 128-row M block, hence every raster band of 16 M blocks
        rows = np.array(rows_per_block(0, M, seed + N), np.int64)
        assert len(rows) >= M // 128
    want = ORC.gemm_nt_rows(p["A"], p["sa"], p["B"], p["sb"], rows)
    U.assert_close(got[rows], want, f"dense {shape}")


@pytest.mark.parametrize("nk", W.GROUPED_NK, ids=lambda s: "x".join(map(str, s)))
def test_contiguous_fullsize(nk):
    N, K = nk
    cfg = W.CONFIGS["grouped_contiguous"]
    p = W.contiguous_problem(cfg["groups"], N, K, *cfg["m_range"], seed=cfg["seed"])
    got = U.run_contiguous(p)
    mi = p["m_indices"]
    pad = mi < 0
    assert np.all(got[pad] == 0)
    assert np.all(np.isfinite(U.bits_to_f64(got[~pad])))
    # every 128-row M block of every expert: one seeded row each, plus the
    # expert's first and last rows
    rows = []
    for e in range(p["G"]):
        r = np.nonzero(mi == e)[0]
        rows += rows_per_block(int(r[0]), int(r[-1]) + 1, 7 + e)
    rows = np.array(sorted(set(rows)), np.int64)
    assert len(rows) >= int(np.sum(mi >= 0)) // 128
    want = ORC.grouped_contiguous(p["A"], p["sa"], p["B"], p["sb"], mi, rows=rows)
    U.assert_close(got[rows], want, f"contiguous {nk}")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("nk", W.GROUPED_NK, ids=lambda s: "x".join(map(str, s)))
def test_masked_fullsize(G, nk):
    N, K = nk
    cfg = W.CONFIGS["grouped_masked"]
    p = W.masked_problem(G, cfg["max_m"], N, K, cfg["expected_m"], seed=cfg["seed"] + G)
    got = U.run_masked(p, expected_m=cfg["expected_m"])
    mm = p["masked_m"]
    rng = np.random.default_rng(G)
    for g in range(G):
        v = int(mm[g])
        assert np.all(got[g, v:] == W.BF16_SENTINEL), f"group {g} rows past {v} written"
        # every 128-row M block of the group's valid rows, plus one more random row
        rows = np.array(sorted({*rows_per_block(0, v, G * 1000 + g),
                                int(rng.integers(0, v))}), np.int64)
        want = ORC.gemm_nt_rows(p["A"][g], p["sa"][g], p["B"][g], p["sb"][g], rows)
        U.assert_close(got[g][rows], want, f"masked G={G} {nk} group {g}")

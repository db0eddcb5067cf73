"""The planner's choices on the benchmark workloads' shapes (host only, no GPU):
the configurations that per-case sweeps of every instance measured best, or
within a few percent of it, stay the ones the time model picks.  Planned as
for 152 SMs with num_sms / S clusters of S CTAs resident (the planner's rule
without a GB300 present)."""
import pytest
import torch

import moe_grouped_gemm_bf16_gb300 as dg
from moe_grouped_gemm_bf16_gb300 import _build

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="with a GPU present the planner uses its occupancy")

DENSE, CONTIGUOUS, MASKED = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    dg.debug_force_config(0, 0)
    dg.debug_force_pair(-1)
    dg.debug_force_block_scaled(-1)


def plan(kind, m, n, k, g=1, ue8m0=False):
    c = dg.plan_config(kind, m, n, k, g, 152, ue8m0=ue8m0)
    return c["block_n"], c["split_k"], c["pair"], c["block_scaled"]


@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
def test_decode_splits_k_over_clusters(ue8m0):
    # few output tiles: the K groups are split; 2112 columns take 64-wide tiles
    assert plan(DENSE, 64, 2112, 7168, ue8m0=ue8m0) == (64, 4, 0, 0)
    assert plan(DENSE, 128, 2112, 7168, ue8m0=ue8m0) == (64, 4, 0, 0)
    assert plan(DENSE, 64, 4096, 7168, ue8m0=ue8m0) == (128, 4, 0, 0)
    assert plan(DENSE, 128, 7168, 16384, ue8m0=ue8m0) == (128, 2, 0, 0)
    # enough N tiles: no split
    assert plan(DENSE, 64, 7168, 2048, ue8m0=ue8m0)[1] == 1


def test_fp32_prefill_and_grouped_take_wide_unsplit_tiles():
    for n, k in ((2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168),
                 (7168, 2048)):
        assert plan(DENSE, 4096, n, k) == (256, 1, 0, 0), (n, k)
    for n, k in ((4096, 7168), (7168, 2048)):
        assert plan(CONTIGUOUS, 34048, n, k, 4) == (256, 1, 0, 0), (n, k)
    # masked: the small groups' few M blocks take narrower tiles
    assert plan(MASKED, 256, 4096, 7168, 1) == (64, 1, 0, 0)
    assert plan(MASKED, 256, 4096, 7168, 8) == (256, 1, 0, 0)


def test_packed_scales_take_the_block_scaled_kernel_for_prefill():
    # one CTA per tile (the CTA pair measured slower); 224-wide tiles where
    # they fill the SMs better
    for n, k in ((2112, 7168), (24576, 1536), (7168, 16384), (7168, 2048)):
        assert plan(DENSE, 4096, n, k, ue8m0=True) == (256, 1, 0, 1), (n, k)
    assert plan(DENSE, 4096, 4096, 7168, ue8m0=True) == (224, 1, 0, 1)
    assert plan(DENSE, 4096, 32768, 512, ue8m0=True) == (224, 1, 0, 1)
    for n, k in ((4096, 7168), (7168, 2048)):
        assert plan(CONTIGUOUS, 34048, n, k, 4, ue8m0=True) == (256, 1, 0, 1), (n, k)
    for g in (4, 8):
        assert plan(MASKED, 256, 7168, 2048, g, ue8m0=True)[3] == 1
    # the smallest masked groups keep the promotion kernels' 64-wide twin
    assert plan(MASKED, 256, 4096, 7168, 1, ue8m0=True) == (64, 1, 0, 0)


def test_pairs_only_when_forced():
    try:
        for ue8m0 in (False, True):
            assert plan(DENSE, 4096, 7168, 7168, ue8m0=ue8m0)[2] == 0
            dg.debug_force_pair(1)
            assert plan(DENSE, 4096, 7168, 7168, ue8m0=ue8m0)[2] == 1
            dg.debug_force_pair(-1)
    finally:
        dg.debug_force_pair(-1)

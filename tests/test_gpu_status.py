"""Device-side error reporting, tested without faulting the GPU:

* out-of-range masked_m values are clamped and flagged;
* a contiguous block that mixes two experts, or an expert id past the group
  count, is flagged and written as zeros;
* the bounded waits: with the TMA producer switched off (a flag that nothing
  sets) and a short time limit, every wait runs out, the kernel finishes,
  reports DG_ERR_TIMEOUT, and the context stays usable for a correct run.
"""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_bf16_gb300 as dg
import oracle
import workloads as W
from moe_grouped_gemm_bf16_gb300 import _build
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DG_OK, DG_ERR_TIMEOUT, DG_ERR_MASK_RANGE, DG_ERR_EXPERT_RANGE = 0, 7, 8, 9


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    torch.cuda.init()
    dg.get_device_status()  # clear
    yield
    dg.debug_set_skip_producer(False)
    dg.set_wait_timeout_ns(0)


def test_status_clean_after_normal_run():
    p = W.dense_problem(128, 256, 512, seed=1)
    U.run_dense(p)
    assert dg.get_device_status() == DG_OK


def test_masked_out_of_range_is_clamped_and_flagged():
    p = W.masked_problem(3, 200, 256, 256, 60, seed=2)
    mm = np.array([-5, 250, 70], np.int32)  # -5 -> 0, 250 -> 200 (= max_m)
    got = U.run_masked(p, masked_m=mm)
    assert dg.get_device_status() == DG_ERR_MASK_RANGE
    assert dg.get_device_status() == DG_OK  # reading clears it
    init = np.full(got.shape, W.BF16_SENTINEL, np.uint16)
    want = oracle.Oracle().grouped_masked(p["A"], p["sa"], p["B"], p["sb"],
                                          np.array([0, 200, 70], np.int32), init)
    assert np.all(got[0] == W.BF16_SENTINEL)
    U.assert_close(got[1], want[1], "clamped to max_m")
    U.assert_close(got[2, :70], want[2, :70], "group 2")
    assert np.all(got[2, 70:] == W.BF16_SENTINEL)


def test_contiguous_bad_expert_ids_are_flagged():
    p = W.contiguous_problem(2, 256, 256, 128, 128, seed=3)  # two full 128-row blocks
    mi = p["m_indices"].copy()
    mi[5] = 1 - mi[0]          # block 0 mixes experts 0 and 1
    mi[128:256] = 7            # block 1 names an expert past num_groups
    p = dict(p, m_indices=mi)
    got = U.run_contiguous(p)
    assert dg.get_device_status() == DG_ERR_EXPERT_RANGE
    assert np.all(got[5] == 0) and np.all(got[128:256] == 0)
    want = oracle.Oracle().grouped_contiguous(p["A"], p["sa"], p["B"], p["sb"], mi, rows=[0, 1, 6])
    U.assert_close(got[[0, 1, 6]], want, "rows of the block's own expert")


def test_wait_timeout_is_reported_and_context_survives():
    p = W.dense_problem(256, 512, 1024, seed=4)
    dg.set_wait_timeout_ns(20_000_000)  # 20 ms
    dg.debug_set_skip_producer(True)
    try:
        U.run_dense(p)
        st = dg.get_device_status()
    finally:
        dg.debug_set_skip_producer(False)
        dg.set_wait_timeout_ns(0)
    assert st == DG_ERR_TIMEOUT
    got = U.run_dense(p)
    assert dg.get_device_status() == DG_OK
    U.assert_close(got, oracle.Oracle().gemm_nt(p["A"], p["sa"], p["B"], p["sb"]), "after timeout")


def test_wait_timeout_split_cluster():
    """Same, in the cluster (K split) configuration."""
    p = W.dense_problem(64, 512, 1024, seed=5)
    dg.set_wait_timeout_ns(20_000_000)
    dg.debug_set_skip_producer(True)
    try:
        with U.forced_config(128, 4):
            U.run_dense(p)
        st = dg.get_device_status()
    finally:
        dg.debug_set_skip_producer(False)
        dg.set_wait_timeout_ns(0)
    assert st == DG_ERR_TIMEOUT
    with U.forced_config(128, 4):
        got = U.run_dense(p)
    assert dg.get_device_status() == DG_OK
    U.assert_close(got, oracle.Oracle().gemm_nt(p["A"], p["sa"], p["B"], p["sb"]), "after timeout")

"""The C-ABI library on the host: it loads, exports what include/dg.h declares,
and rejects bad arguments before launching anything.  No GPU needed: argument
errors are found before the library touches a device."""
import ctypes
import os
import re

import pytest

import moe_grouped_gemm_bf16_gb300 as dg
from moe_grouped_gemm_bf16_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return dg.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    decl = declared_functions()
    assert len(decl) >= 14
    for name in decl:
        assert hasattr(L, name), name
    assert sorted(decl) == sorted(dg.EXPORTED_SYMBOLS)


# a fake, 16-byte aligned "device" address: never dereferenced by these tests
P = 0x10000


def _dense(**kw):
    a = dict(A=P, sa=P, ld_sa=128, B=P, sb=P, D=P, M=128, N=256, K=512)
    a.update(kw)
    return a


def status_of(fn, **kw):
    try:
        fn(**kw)
    except dg.DGError as e:
        return e.status
    return 0


@pytest.mark.parametrize("kw,code", [
    (dict(A=None), 1),
    (dict(D=None), 1),
    (dict(M=-1), 1),
    (dict(K=500), 2),
    (dict(K=0), 2),
    (dict(K=128 * 513), 2),
    (dict(N=200), 2),
    (dict(N=8), 2),
    (dict(A=P + 8), 3),
    (dict(D=P + 2), 3),
    (dict(sa=P + 4), 3),
    (dict(ld_sa=130), 3),
    (dict(ld_sa=64), 1),
])
def test_dense_argument_errors(L, kw, code):
    assert status_of(dg.gemm_fp8_fp8_bf16_nt, **_dense(**kw)) == code
    assert dg.lib().dg_last_error_string().decode() != ""


def test_add_c_requires_c(L):
    a = _dense()
    assert status_of(dg.gemm_fp8_fp8_bf16_nt_add_c, C=None, **a) == 1
    assert status_of(dg.gemm_fp8_fp8_bf16_nt_add_c, C=P + 8, **a) == 3


@pytest.mark.parametrize("name", ["nn", "tn", "tt"])
def test_layout_argument_errors(L, name):
    fn = getattr(dg, "gemm_fp8_fp8_bf16_" + name)
    a_t = name[0] == "t"
    assert status_of(fn, **_dense(A=None)) == 1
    assert status_of(fn, **_dense(K=500)) == 2
    assert status_of(fn, **_dense(N=200)) == 2
    assert status_of(fn, **_dense(C=P + 8)) == 3
    assert status_of(fn, **_dense(ld_sa=64)) == 1
    # A stored [K][M]: a row is M bytes, so M must keep TMA's 16-byte pitch
    assert (status_of(fn, **_dense(M=120, ld_sa=120)) == 2) == a_t
    assert status_of(fn, **_dense(M=0)) == 0


def _kg(**kw):
    a = dict(A=P, sa=P, ld_sa=256, B=P, sb=P, D=P, ks=P, num_groups=4, M=256, N=512,
             K_total=2048)
    a.update(kw)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(A=None), 1),
    (dict(ks=None), 1),
    (dict(num_groups=0), 1),
    (dict(num_groups=1025), 1),
    (dict(ld_sa=128), 1),
    (dict(K_total=500), 2),
    (dict(K_total=0), 2),
    (dict(K_total=128 * 513), 2),
    (dict(M=120, ld_sa=120), 2),
    (dict(N=200), 2),
    (dict(C=P + 8), 3),
    (dict(ks=P + 2), 3),
    (dict(ld_sa=258), 3),
    (dict(M=0), 0),
])
def test_k_grouped_argument_errors(L, kw, code):
    assert status_of(dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous, **_kg(**kw)) == code


def test_ue8m0_argument_errors(L):
    d = dict(A=P, sfa=P, ld_sfa=128, B=P, sfb=P, D=P, M=128, N=256, K=512)
    f = dg.gemm_fp8_fp8_bf16_nt_ue8m0
    assert status_of(f, **{**d, "sfa": None}) == 1
    assert status_of(f, **{**d, "ld_sfa": 64}) == 1
    assert status_of(f, **{**d, "ld_sfa": 130}) == 3
    assert status_of(f, **{**d, "sfa": P + 4}) == 3
    assert status_of(f, **{**d, "sfb": P + 2}) == 3
    assert status_of(f, **{**d, "K": 500}) == 2
    assert status_of(f, **{**d, "M": 0}) == 0
    c = dict(A=P, sfa=P, ld_sfa=256, B=P, sfb=P, D=P, m_indices=P, M_total=256, N=256, K=512,
             num_groups=4)
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0, **{**c, "m_indices": None}) == 1
    m = dict(A=P, sfa=P, ld_sfa=128, B=P, sfb=P, D=P, masked_m=P, num_groups=4, max_m=128, N=256,
             K=512, expected_m=64)
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0, **{**m, "num_groups": 1025}) == 1
    q = dict(X=P, Q=P, sfa=P, num_groups=1, M=128, K=512, ld_sfa=128)
    assert status_of(dg.quantize_fp8_1x128_ue8m0, **{**q, "sfa": None}) == 1
    assert status_of(dg.quantize_fp8_1x128_ue8m0, **{**q, "K": 200}) == 2
    assert status_of(dg.quantize_fp8_1x128_ue8m0, **{**q, "ld_sfa": 130}) == 3
    assert status_of(dg.quantize_fp8_1x128_ue8m0, **{**q, "M": 0, "ld_sfa": 0}) == 0


@pytest.mark.parametrize("name", ["nn", "tn", "tt"])
def test_layout_ue8m0_argument_errors(L, name):
    fn = getattr(dg, f"gemm_fp8_fp8_bf16_{name}_ue8m0")
    d = dict(A=P, sfa=P, ld_sfa=128, B=P, sfb=P, D=P, M=128, N=256, K=512)
    assert status_of(fn, **{**d, "sfa": None}) == 1
    assert status_of(fn, **{**d, "K": 500}) == 2
    assert status_of(fn, **{**d, "ld_sfa": 130}) == 3
    assert status_of(fn, **{**d, "C": P + 8}) == 3
    assert (status_of(fn, **{**d, "M": 120, "ld_sfa": 120}) == 2) == (name[0] == "t")
    assert status_of(fn, **{**d, "M": 0}) == 0


def test_k_grouped_ue8m0_argument_errors(L):
    f = dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0
    d = dict(A=P, sfa=P, ld_sfa=256, B=P, sfb=P, D=P, ks=P, num_groups=4, M=256, N=512,
             K_total=2048)
    assert status_of(f, **{**d, "ks": None}) == 1
    assert status_of(f, **{**d, "num_groups": 1025}) == 1
    assert status_of(f, **{**d, "K_total": 500}) == 2
    assert status_of(f, **{**d, "M": 120, "ld_sfa": 120}) == 2
    assert status_of(f, **{**d, "sfb": P + 2}) == 3
    assert status_of(f, **{**d, "M": 0}) == 0


def test_empty_problem_is_a_noop(L):
    # M = 0: nothing to compute, no device needed
    assert status_of(dg.gemm_fp8_fp8_bf16_nt, **_dense(M=0)) == 0


def test_grouped_argument_errors(L):
    c = dict(A=P, sa=P, ld_sa=256, B=P, sb=P, D=P, m_indices=P, M_total=256, N=256, K=512,
             num_groups=4)
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous, **{**c, "M_total": 200,
                                                                        "ld_sa": 200}) == 2
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous, **{**c, "num_groups": 0}) == 1
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_contiguous, **{**c, "m_indices": None}) == 1
    m = dict(A=P, sa=P, ld_sa=128, B=P, sb=P, D=P, masked_m=P, num_groups=4, max_m=128, N=256,
             K=512, expected_m=64)
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked, **{**m, "num_groups": 1025}) == 1
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked, **{**m, "masked_m": None}) == 1
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked, **{**m, "ld_sa": 100}) == 1
    assert status_of(dg.m_grouped_gemm_fp8_fp8_bf16_nt_masked, **{**m, "max_m": 0}) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(X=None), 1),
    (dict(sa=None), 1),
    (dict(num_groups=0), 1),
    (dict(M=-1), 1),
    (dict(ld_sa=64), 1),
    (dict(K=200), 2),
    (dict(K=0), 2),
    (dict(num_groups=1 << 12, M=1 << 12, K=128 * 256, ld_sa=1 << 12), 2),
    (dict(ld_sa=130), 3),
    (dict(X=P + 8), 3),
    (dict(Q=P + 4), 3),
])
def test_quantiser_argument_errors(L, kw, code):
    a = dict(X=P, Q=P, sa=P, num_groups=1, M=128, K=512, ld_sa=128)
    a.update(kw)
    assert status_of(dg.quantize_fp8_1x128, **a) == code
    assert dg.lib().dg_last_error_string().decode() != ""


def test_quantiser_empty_is_a_noop(L):
    assert status_of(dg.quantize_fp8_1x128, X=P, Q=P, sa=P, num_groups=1, M=0, K=512,
                     ld_sa=0) == 0


def test_valid_call_without_device_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert status_of(dg.gemm_fp8_fp8_bf16_nt, **_dense()) in (4,)


def test_utilities(L):
    assert dg.get_mk_alignment_for_contiguous_layout() == 128
    # fp32 scales: 4 elements per 16 bytes
    assert [dg.get_tma_aligned_size(m, 4) for m in (0, 1, 4, 5, 64, 130)] == [0, 4, 4, 8, 64, 132]
    assert dg.get_tma_aligned_size(7, 2) == 8
    assert dg.get_tma_aligned_size(17, 1) == 32
    assert dg.get_tma_aligned_size(-1, 4) == -1
    with pytest.raises(dg.DGError):
        dg.set_num_sms(-3)
    dg.set_wait_timeout_ns(0)


def test_sm_fill_golden(L):
    """The pages' unaligned-block-size example: tile counts (one tile per SM)."""
    rows = []
    with open(os.path.join(GOLDEN, "sm_fill_example.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].split()
            if line:
                rows.append([int(x) for x in line])
    assert len(rows) == 2
    for M, N, bm, bn, tiles in rows:
        assert dg.num_output_tiles(M, N, bm, bn) == tiles


def test_plan_config_heuristic(L):
    # decode: few output tiles -> the K groups are split over a cluster
    cfg = dg.plan_config(0, 64, 2112, 7168, 1, 152)
    assert cfg["split_k"] > 1 and cfg["grid"] <= 152 and cfg["block_m"] == 128
    # prefill: enough tiles -> no split, wide tiles
    cfg = dg.plan_config(0, 4096, 7168, 7168, 1, 152)
    assert cfg["split_k"] == 1 and cfg["grid"] <= 152
    assert cfg["num_tiles"] == (4096 // cfg["block_m"]) * ((7168 + cfg["block_n"] - 1) // cfg["block_n"])
    assert cfg["block_m"] == (256 if cfg["pair"] else 128)
    # the pair form is for M > 128 only (unless forced)
    assert dg.plan_config(0, 128, 7168, 7168, 1, 152)["pair"] == 0
    for kind, m, g in ((1, 32768, 4), (2, 256, 8)):
        cfg = dg.plan_config(kind, m, 4096, 7168, g, 152)
        assert cfg["split_k"] == 1 and cfg["smem_bytes"] <= 232448
    # K-grouped: one tile set per group, no split, MN-major instances
    cfg = dg.plan_config(3, 4096, 7168, 4 * 4096, 4, 152)
    assert cfg["split_k"] == 1 and cfg["pair"] == 0 and cfg["smem_bytes"] <= 232448
    assert cfg["num_tiles"] == 4 * 32 * ((7168 + cfg["block_n"] - 1) // cfg["block_n"])
    with pytest.raises(dg.DGError):
        dg.plan_config(0, 64, 2112, 7000, 1, 152)
    with pytest.raises(dg.DGError):
        dg.plan_config(4, 64, 2112, 7168, 1, 152)
    with pytest.raises(dg.DGError):
        dg.plan_config(4, 64, 2112, 7168, 1, 152, ue8m0=True)
    # the fp32-scale entry points have no block-scaled kernel
    for kind, m, g in ((0, 4096, 1), (1, 32768, 4), (2, 256, 8), (0, 64, 1)):
        assert dg.plan_config(kind, m, 7168, 7168, g, 152)["block_scaled"] == 0
    # packed UE8M0 scales: the block-scaled kernel for prefill and the grouped
    # prefill shapes; decode keeps the promotion kernels' K split
    for kind, m, g in ((0, 4096, 1), (1, 32768, 4), (2, 256, 8)):
        cfg = dg.plan_config(kind, m, 7168, 7168, g, 152, ue8m0=True)
        assert cfg["block_scaled"] == 1 and cfg["split_k"] == 1, (kind, cfg)
    cfg = dg.plan_config(0, 64, 7168, 7168, 1, 152, ue8m0=True)
    assert cfg["block_scaled"] == 0 and cfg["split_k"] > 1


def test_force_config_hook(L):
    try:
        dg.debug_force_pair(1)
        assert dg.plan_config(0, 4096, 4096, 1024, 1, 152)["pair"] == 1
        dg.debug_force_pair(0)
        assert dg.plan_config(0, 4096, 4096, 1024, 1, 152)["pair"] == 0
        dg.debug_force_pair(-1)
        dg.debug_force_config(256, 0)
        assert dg.plan_config(0, 4096, 4096, 1024, 1, 152)["block_n"] == 256
        dg.debug_force_config(128, 4)
        cfg = dg.plan_config(0, 128, 4096, 1024, 1, 152)
        assert (cfg["block_n"], cfg["split_k"]) == (128, 4)
        with pytest.raises(dg.DGError):
            dg.debug_force_config(128, 9)
    finally:
        dg.debug_force_config(0, 0)
        dg.debug_force_pair(-1)


def test_checked_build_exports_every_declared_symbol():
    """The checked library (every kernel compiled with DG_DEBUG=1) builds on
    a machine without a GPU and exports the same ABI."""
    path = _build.build(debug=True)
    assert os.path.basename(path) == "libdg_debug.so"
    Ld = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(Ld, name), name

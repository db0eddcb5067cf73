"""Host logic of bench.py that needs no GPU: the source hash that ties a
committed ncu traffic record to the code it was taken on ignores comments and
blank space, changes with the code, and the algorithmic counts of a case
follow the stated formulas."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_code_only_ignores_comments_and_space():
    b = _bench()
    a = "int x = 1; // one\n/* block\n comment */ int y=2;\n"
    c = "int x = 1;\n\n   int y=2;   // other words\n"
    assert b._code_only(a) == b._code_only(c)
    assert b._code_only("int x = 1;") != b._code_only("int x = 2;")


def test_kernel_source_hash_is_stable_and_per_workload():
    b = _bench()
    h1, h2 = b.kernel_source_hash("dense_decode"), b.kernel_source_hash("dense_decode")
    assert h1 == h2 and len(h1) == 16
    assert b.kernel_source_hash("quantize_act") != h1


def test_case_algorithmic_counts():
    b = _bench()
    M, N, K = 64, 300, 512
    p = dict(A=None, M=M, N=N, K=K)
    c = b.Case("dense", p, "x")
    kb, nb = K // 128, (N + 127) // 128
    assert c.flops == 2.0 * M * N * K
    assert c.bytes == M * K + N * K + 4 * M * kb + 4 * nb * kb + 2 * M * N
    ks = np.array([256, 0, 384], np.int32)
    q = dict(M=M, N=N, K=int(ks.sum()), G=3, ks=ks)
    k = b.Case("k_grouped", q, "y")
    Kt = int(ks.sum())
    assert k.flops == 2.0 * M * N * Kt
    assert k.bytes == Kt * M + Kt * N + 4 * M * (Kt // 128) + 4 * nb * (Kt // 128) + 2 * 3 * M * N


def test_ue8m0_stand_in_scales():
    """The bench's packed UE8M0 stand-ins decode (through the oracle) to the
    fp32 values the generator reports, each the power-of-two ceiling of the
    original scale."""
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import workloads as W
    p = W.dense_problem(40, 300, 640, seed=3)
    sfa, sfb, sa2, sb2 = W.ue8m0_packed_scales(p["sa"], p["sb"])
    orc = oracle.Oracle()
    kb = 640 // 128
    assert np.array_equal(orc.decode_sfa(sfa, kb), sa2)
    assert np.array_equal(orc.decode_sfb(sfb, kb), sb2)
    live = p["sa"][:, :40]
    assert np.all(sa2[:, :40] >= live) and np.all(sa2[:, :40] < 2 * live)
    assert np.all(sb2 >= p["sb"]) and np.all(sb2 < 2 * p["sb"])
    assert np.all(np.log2(sb2) == np.round(np.log2(sb2)))


def _fake(b, bytes_, flops):
    c = b.Case("dense", dict(A=None, M=64, N=128, K=128), "f")
    c.bytes, c.flops = bytes_, flops
    return c


def test_binding_roof_fractions():
    """Each case is judged against the roof it is bound by: its ideal time is
    the larger of bytes / HBM peak and FLOPs / FP8 peak, and a step's
    fraction is the sum of the ideal times over the measured time."""
    b = _bench()
    pk = b.Peaks()
    pk.hbm, pk.fp8 = 1000.0, 2000.0          # GB/s, TFLOP/s
    mem = _fake(b, 1e9, 1e12)                # 1 ms of HBM, 0.5 ms of tensor
    cmp_ = _fake(b, 1e8, 4e12)               # 0.1 ms of HBM, 2 ms of tensor
    assert abs(pk.ideal_s(mem) - 1e-3) < 1e-12 and abs(pk.ideal_s(cmp_) - 2e-3) < 1e-12
    assert pk.bound([mem]) == "hbm" and pk.bound([cmp_]) == "tensor"
    assert pk.bound([mem, cmp_]) == "tensor"   # 1.1 ms of HBM against 2.5 ms of tensor
    r = b.roofline("none", [mem, cmp_], 6e-3, pk, 2)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 5e12 / 6e-3 / 1e12) < 0.1
    assert abs(r["frac"] - (5e12 / 6e-3 / 1e12) / 2000.0) < 1e-4
    assert abs(r["frac_binding"] - 0.5) < 1e-4            # (1 + 2) ms ideal over 6 ms
    assert r["cases_hbm_bound"] == 1 and r["cases_tensor_bound"] == 1
    nom = max(1e9 / 8000e9, 1e12 / 4500e12) + max(1e8 / 8000e9, 4e12 / 4500e12)
    assert abs(r["frac_binding_nominal"] - nom / 6e-3) < 1e-4
    assert abs(b.value_of([mem, cmp_], 2.0, "GB/s") - 1.1e9 / 2.0 / 1e9) < 1e-9


def test_oracle_sample_shape_fits_the_budget():
    """A case's oracle sample takes whole rows (a multiple of the core count)
    once a row block of all columns fits the budget, and never more rows than
    the case has."""
    b = _bench()
    c = b.Case("dense", dict(A=None, M=4096, N=1024, K=1024), "d")
    rows, cols = b._sample_shape(c, 1.0, 1e9, 8)           # 1e9 MACs: ~950 rows of 1M MACs
    assert cols == 1024 and rows % 8 == 0 and rows * 1024 * 1024 <= 1e9
    rows, cols = b._sample_shape(c, 1e-3, 1e9, 8)          # 1e6 MACs: 8 rows x ~120 columns
    assert rows == 8 and cols % 16 == 0 and cols < 1024
    rows, cols = b._sample_shape(c, 1e6, 1e9, 8)
    assert rows == 4096 and cols == 1024


def test_nvml_sampler_summary_reads_reason_bits():
    """The NVML clock record: median SM clock of the reads inside the region,
    the clock-event reasons from their bits, power in W."""
    import bench
    s = bench.NvmlSampler(0)
    s.max_mhz = 2070.0
    s.samples = [(1.0, 2070.0, 0, 900000), (2.0, 2000.0, 0x4, 1200000), (3.0, 1990.0, 0x4, 1300000),
                 (9.0, 1000.0, 0x8 | 0x40, 100000)]
    rec = s.summarize(0.5, 3.5)
    assert rec["sm_mhz"] == 2000.0 and rec["samples"] == 3 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["power_w_max"] == 1300.0
    assert s.summarize(8.5, 9.5)["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert s.summarize(20, 30) is None

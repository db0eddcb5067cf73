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

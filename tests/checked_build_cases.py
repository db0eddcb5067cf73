"""Small cases of every form of the GEMM, run through whichever library the
binding loaded, each compared with the CPU oracle and followed by a read of
the device status word.  Run by tests/test_gpu_checked_build.py in a child
process with DG_DEBUG=1, so that the checked library (bounds checks before
each TMA load and plain global store, fill checks after each ring wait) is
the one loaded; prints "checked ok" and the library's path at the end."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_grouped_gemm_bf16_gb300 as dg  # noqa: E402
import oracle  # noqa: E402
import workloads as W  # noqa: E402
from tests import gpu_util as U  # noqa: E402
from tests.test_gpu_ue8m0 import dense_ue8m0  # noqa: E402


def status_ok(what):
    torch.cuda.synchronize()
    st = dg.get_device_status()
    assert st == 0, f"{what}: device status {dg.STATUS_NAMES.get(st, st)}"


def main():
    orc = oracle.Oracle()
    torch.cuda.set_device(0)
    # dense nt: heuristic, forced K split, 64-row A, CTA pair; ragged edges
    for M, N, K, cfg in [(200, 400, 1152, (0, 0, -1)), (64, 2112, 2048, (128, 3, -1)),
                         (64, 512, 1024, (128, 4, -1)), (300, 528, 640, (256, 1, 1))]:
        p = W.dense_problem(M, N, K, seed=M + N)
        with U.forced_config(*cfg):
            got = U.run_dense(p)
            status_ok(f"dense {M}x{N}x{K} {cfg}")
        U.assert_close(got, orc.gemm_nt(p["A"], p["sa"], p["B"], p["sb"]), f"dense {cfg}")
    # contiguous (a padding block, ragged expert segments)
    q = W.contiguous_problem(3, 400, 1152, 100, 300, seed=8)
    got = U.run_contiguous(q)
    status_ok("contiguous")
    want = orc.grouped_contiguous(q["A"], q["sa"], q["B"], q["sb"], q["m_indices"])
    pad = q["m_indices"] < 0
    assert np.all(got[pad] == 0)
    U.assert_close(got[~pad], want[~pad], "contiguous")
    # masked, plain and over CTA pairs (an empty group and a partial block)
    for pair in (0, 1):
        mm = np.array([0, 1, 129, 256], np.int32)
        r = W.masked_problem(4, 256, 528, 1152, 90, seed=12)
        with U.forced_config(0, 0, pair=pair):
            got = U.run_masked(r, masked_m=mm, expected_m=90)
            status_ok(f"masked pair={pair}")
        init = np.full(got.shape, W.BF16_SENTINEL, np.uint16)
        want = orc.grouped_masked(r["A"], r["sa"], r["B"], r["sb"], mm, init)
        for g in range(4):
            v = int(mm[g])
            assert np.array_equal(got[g, v:], want[g, v:])
            U.assert_close(got[g, :v], want[g, :v], f"masked pair={pair} group {g}")
    # tn with an addend, and the K-grouped form with an empty group
    p = W.dense_problem(208, 400, 1152, seed=3)
    At, Bt = np.ascontiguousarray(p["A"].T), np.ascontiguousarray(p["B"].T)
    C = torch.randn(208, 400).to(torch.bfloat16)
    D = torch.empty((208, 400), dtype=torch.bfloat16, device="cuda")
    dg.gemm_fp8_fp8_bf16_tn(U.dev(At), U.dev(p["sa"]), p["sa"].shape[-1], U.dev(Bt),
                            U.dev(p["sb"]), D, 208, 400, 1152, C=C.cuda())
    status_ok("tn + C")
    Cb = C.view(torch.int16).numpy().view(np.uint16)
    U.assert_close(U.to_bits(D), orc.gemm_layout("tn", At, p["sa"], Bt, p["sb"], Cb), "tn")
    kg = W.k_grouped_problem([256, 0, 384], 128, 256, seed=6)
    Dk = torch.empty((3, 128, 256), dtype=torch.bfloat16, device="cuda")
    dg.k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(U.dev(kg["A"]), U.dev(kg["sa"]),
                                                 kg["sa"].shape[-1], U.dev(kg["B"]),
                                                 U.dev(kg["sb"]), Dk, U.dev(kg["ks"]), 3, 128,
                                                 256, kg["K"])
    status_ok("k-grouped")
    want = orc.k_grouped_tn(kg["A"], kg["sa"], kg["B"], kg["sb"], kg["ks"])
    for g in range(3):
        U.assert_close(U.to_bits(Dk[g]), want[g], f"k-grouped {g}")
    # packed UE8M0 scales: the block-scaled kernels (plain and CTA pair) and
    # the promotion kernels
    for bs, pair in ((1, 0), (1, 1), (0, 0)):
        u = dense_ue8m0(333, 528, 896, seed=9)
        dg.debug_force_block_scaled(bs)
        A, B = U.dev(u["A"]), U.dev(u["B"])
        D = torch.full((333, 528), -1, dtype=torch.int16, device="cuda")
        with U.forced_config(0, 0, pair=pair):
            dg.gemm_fp8_fp8_bf16_nt_ue8m0(A, U.dev(u["sfa"]), u["sfa"].shape[-1], B,
                                          U.dev(u["sfb"]), D, 333, 528, 896)
            status_ok(f"ue8m0 block_scaled={bs} pair={pair}")
        dg.debug_force_block_scaled(-1)
        U.assert_close(U.to_bits(D), orc.gemm_nt_ue8m0(u["A"], u["sfa"], u["B"], u["sfb"]),
                       f"ue8m0 block_scaled={bs} pair={pair}")
    print("checked ok", dg.lib()._name)


if __name__ == "__main__":
    main()

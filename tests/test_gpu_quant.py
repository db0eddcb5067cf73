"""The CUDA activation quantiser against the CPU oracle, bit for bit (codes and
scales are exact functions of the bf16 input in fp32), through the C ABI; and
the chain quantiser -> GEMM against the oracle's quantiser -> GEMM."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_bf16_gb300 as dg
import oracle
from moe_grouped_gemm_bf16_gb300 import _build
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

ORC = None
SA_FILL = np.float32(-7.25)  # the value scale columns past M must keep


@pytest.fixture(scope="module", autouse=True)
def built():
    global ORC
    _build.build()
    ORC = oracle.Oracle()
    torch.cuda.init()


def make_input(G, M, K, seed):
    """bf16 bits [G,M,K]: normal values with a per-group magnitude spread over
    60 binades, plus edge groups (all zero, below the 1e-4 floor, bf16 values
    near the top and bottom of the range, negative zeros)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(G, M, K, generator=g, dtype=torch.float32)
    mag = torch.randint(-30, 30, (G, M, K // 128), generator=g).to(torch.float32)
    x *= torch.exp2(mag).repeat_interleave(128, dim=-1)
    if M >= 4 and K >= 256:
        x[0, 0, :128] = 0.0
        x[0, 1, 128:256] = 3e-7 * torch.sign(x[0, 1, 128:256])
        x[0, 2, :128] = torch.randn(128, generator=g) * 1e30
        x[0, 3, :128] = -0.0
        x[0, 3, 5] = 1e-35
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def run_gpu(bits, ld_sa):
    G, M, K = bits.shape
    X = torch.from_numpy(bits.view(np.int16)).cuda()
    Q = torch.empty((G, M, K), dtype=torch.uint8, device="cuda")
    sa = torch.full((G, K // 128, ld_sa), float(SA_FILL), dtype=torch.float32, device="cuda")
    dg.quantize_fp8_1x128(X, Q, sa, G, M, K, ld_sa)
    torch.cuda.synchronize()
    return Q.cpu().numpy(), sa.cpu().numpy()


def check(bits, ld_sa, what):
    Q, sa = run_gpu(bits, ld_sa)
    Qr, sar = ORC.quantize_1x128(bits, ld_sa=ld_sa, sa_fill=SA_FILL)
    M = bits.shape[1]
    bad = np.argwhere(Q != Qr)
    assert bad.size == 0, f"{what}: {len(bad)} codes differ, first {bad[:4].tolist()}"
    assert np.array_equal(sa[:, :, :M].view(np.uint32), sar[:, :, :M].view(np.uint32)), \
        f"{what}: scales differ"
    assert np.all(sa[:, :, M:] == SA_FILL), f"{what}: scale columns past M written"


SHAPES = [
    (1, 1, 128, 4),       # one unit
    (1, 37, 256, 40),     # ragged M, padded ld_sa
    (1, 200, 1024, 200),
    (3, 65, 384, 68),     # batch of groups (masked layout)
    (2, 1024, 7168, 1024),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_quantiser_matches_oracle(shape):
    G, M, K, ld_sa = shape
    check(make_input(G, M, K, seed=G * 1000 + M + K), ld_sa, f"{shape}")


def test_quantiser_full_size():
    """The prefill activation shape, every code and scale."""
    check(make_input(1, 4096, 7168, seed=77), 4096, "4096x7168")


def test_quantiser_then_gemm():
    """GPU quantiser feeding the GPU GEMM equals the oracle's quantiser feeding
    the oracle's GEMM (same codes and scales, so the GEMM tolerance applies)."""
    M, N, K = 200, 384, 1024
    g = torch.Generator().manual_seed(6)
    xa = torch.randn(M, K, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    B = torch.randint(0, 256, (N, K), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    B = np.where((B & 0x7F) == 0x7F, np.uint8(0), B).astype(np.uint8)
    sb = (torch.rand(((N + 127) // 128, K // 128), generator=g) + 0.5).numpy().astype(np.float32)
    ld_sa = dg.get_tma_aligned_size(M, 4)
    X = torch.from_numpy(xa.view(np.int16)).cuda()
    Q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.zeros((K // 128, ld_sa), dtype=torch.float32, device="cuda")
    dg.quantize_fp8_1x128(X, Q, sa, 1, M, K, ld_sa)
    Bd, sbd = U.dev(B), U.dev(sb)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dg.gemm_fp8_fp8_bf16_nt(Q, sa, ld_sa, Bd, sbd, D, M, N, K)
    torch.cuda.synchronize()
    Qr, sar = ORC.quantize_1x128(xa, ld_sa=ld_sa, sa_fill=0.0)
    want = ORC.gemm_nt(Qr, sar, B, sb)
    U.assert_close(U.to_bits(D), want, "quantise -> gemm")

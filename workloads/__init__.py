"""Seeded synthetic inputs for the FP8 fine-grained-scaled GEMM.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and bench, and holds none of the GEMM's arithmetic: it only draws values and
quantises them into the input format the GEMM takes.

Input format (DeepGEMM, es.news.hada.io/topic?id=19459, "Interfaz GEMM y
restricciones de layout"; fine-grained scaling of DeepSeek-V3 as summarised on
es.news.hada.io/topic?id=19444):
  A  e4m3 [M, K], one fp32 scale per row per 128-wide K group (1x128),
     the scales stored transposed and TMA-aligned: sa[kb, ld_sa], ld_sa = M
     rounded up to a multiple of 4 (16 bytes);
  B  e4m3 [N, K], one fp32 scale per 128x128 block: sb[ceil(N/128), kb].

Recipe: values are fp32 N(0,1) from `torch.Generator().manual_seed(seed)` on
the CPU.  Each 1x128 (A) or 128x128 (B) block is quantised with
scale = max(amax, 1e-4) / 448 and q = e4m3(clamp(x / scale, -448, 448)) using
torch's fp32 -> float8_e4m3fn conversion.  The bytes are produced once and
handed to both sides, so the quantiser's own rounding cannot affect parity.

The workloads are the DeepSeek-V3/R1 inference shapes the pages benchmark
(es.news.hada.io/topic?id=19444, "Rendimiento de GEMM general" and
"Rendimiento de GEMM agrupado para modelos MoE"): no public dataset is
involved; these seeded tensors of the same shapes stand in for them.
"""
import math

import numpy as np
import torch

E4M3_MAX = 448.0
GROUP_K = 128
SCALE_FLOOR = 1e-4

#: (N, K) pairs of the dense decode and prefill sweeps.
DENSE_NK = [(2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048)]
#: (N, K) pairs of the grouped sweeps.
GROUPED_NK = [(4096, 7168), (7168, 2048)]


def align_up(x, a):
    return (x + a - 1) // a * a


def tma_aligned_ld(m):
    """Leading dimension of the transposed activation scales: M rounded up to
    a multiple of 4 floats (16 bytes)."""
    return align_up(m, 4)


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _to_e4m3_bytes(x):
    x = torch.clamp(x, -E4M3_MAX, E4M3_MAX)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def quantize_lhs(x, ld_sa=None):
    """x: float32 [..., M, K] -> (codes uint8 [..., M, K], sa float32 [..., kb, ld_sa]).

    One scale per row per 128-wide K group, stored K-group-major (transposed)."""
    *lead, M, K = x.shape
    assert K % GROUP_K == 0
    kb = K // GROUP_K
    ld_sa = ld_sa or tma_aligned_ld(M)
    xb = x.reshape(*lead, M, kb, GROUP_K)
    amax = xb.abs().amax(dim=-1).clamp_min(SCALE_FLOOR)          # [..., M, kb]
    scale = (amax / E4M3_MAX).to(torch.float32)
    q = _to_e4m3_bytes(xb / scale.unsqueeze(-1)).reshape(*lead, M, K)
    sa = torch.zeros(*lead, kb, ld_sa, dtype=torch.float32)
    sa[..., :M] = scale.transpose(-1, -2)
    return q.contiguous(), sa.contiguous()


def quantize_rhs(x):
    """x: float32 [..., N, K] -> (codes uint8 [..., N, K], sb float32 [..., nb, kb]).

    One scale per 128x128 block; a partial last block of rows uses the amax of
    the rows it has."""
    *lead, N, K = x.shape
    assert K % GROUP_K == 0
    kb = K // GROUP_K
    nb = math.ceil(N / 128)
    pad = nb * 128 - N
    xp = torch.nn.functional.pad(x, (0, 0, 0, pad)) if pad else x
    xb = xp.reshape(*lead, nb, 128, kb, GROUP_K)
    amax = xb.abs().amax(dim=(-3, -1)).clamp_min(SCALE_FLOOR)    # [..., nb, kb]
    scale = (amax / E4M3_MAX).to(torch.float32)
    q = _to_e4m3_bytes(xb / scale[..., :, None, :, None]).reshape(*lead, nb * 128, K)
    return q[..., :N, :].contiguous(), scale.contiguous()


def dense_problem(M, N, K, seed):
    """A dense NT problem.  Returns numpy arrays: A [M,K] u8, sa [kb,ld_sa] f32,
    B [N,K] u8, sb [nb,kb] f32."""
    g = _gen(seed)
    a = torch.randn(M, K, generator=g, dtype=torch.float32)
    b = torch.randn(N, K, generator=g, dtype=torch.float32)
    A, sa = quantize_lhs(a)
    B, sb = quantize_rhs(b)
    return dict(A=A.numpy(), sa=sa.numpy(), B=B.numpy(), sb=sb.numpy(), M=M, N=N, K=K)


def contiguous_problem(num_groups, N, K, m_lo, m_hi, seed, align=128):
    """M-grouped contiguous problem: expert e has m_e ~ U{m_lo..m_hi} rows,
    its segment padded to a multiple of `align` rows.  Padding rows of A hold
    random e4m3 codes (so that zeroing them is really checked) and m_indices
    holds the expert id per row, -1 on padding rows."""
    g = _gen(seed)
    ms = torch.randint(m_lo, m_hi + 1, (num_groups,), generator=g).tolist()
    seg = [align_up(m, align) for m in ms]
    M = sum(seg)
    a = torch.randn(M, K, generator=g, dtype=torch.float32)
    b = torch.randn(num_groups, N, K, generator=g, dtype=torch.float32)
    A, sa = quantize_lhs(a)
    B, sb = quantize_rhs(b)
    m_indices = np.full(M, -1, np.int32)
    off = 0
    for e, (m, s) in enumerate(zip(ms, seg)):
        m_indices[off:off + m] = e
        off += s
    return dict(A=A.numpy(), sa=sa.numpy(), B=B.numpy(), sb=sb.numpy(), m_indices=m_indices,
                M=M, N=N, K=K, G=num_groups, ms=ms)


def k_grouped_problem(ks, M, N, seed):
    """K-grouped (MoE weight-gradient) problem: group g owns ks[g] rows of K
    (multiples of 128, zeros allowed).  The logical operands a [M, K_all] and
    b [N, K_all] are quantised like the dense ones (a per row and 128-wide K
    group, b per 128x128 block) and stored transposed: A [K_all, M],
    B [K_all, N] (the "tn" storage)."""
    ks = np.asarray(ks, np.int32)
    K_all = int(ks.sum())
    g = _gen(seed)
    a = torch.randn(M, K_all, generator=g, dtype=torch.float32)
    b = torch.randn(N, K_all, generator=g, dtype=torch.float32)
    A, sa = quantize_lhs(a)
    B, sb = quantize_rhs(b)
    return dict(A=np.ascontiguousarray(A.numpy().T), sa=sa.numpy(),
                B=np.ascontiguousarray(B.numpy().T), sb=sb.numpy(), ks=ks, M=M, N=N,
                K=K_all, G=len(ks))


def ue8m0_packed_scales(sa, sb):
    """Power-of-two stand-ins for a problem's fp32 scales in the packed UE8M0
    layout (4 K groups per int32, first group in the lowest byte): each scale's
    exponent code, rounded up to the next power of two.  Returns (sfa, sfb,
    sa2, sb2), the last two the fp32 values the codes stand for.
    sa [..., kb, ld] -> sfa [..., ceil(kb/4), ld]; sb [..., nb, kb] -> sfb
    [..., nb, ceil(kb/4)]."""
    def codes(x):
        b = np.ascontiguousarray(x, np.float32).view(np.uint32)
        e = ((b >> 23) & 0xFF) + ((b & 0x7FFFFF) != 0)
        return np.where(x > 0, e, 127).astype(np.uint8)

    def pack(c):
        pad = (-c.shape[-1]) % 4
        if pad:
            c = np.concatenate([c, np.zeros(c.shape[:-1] + (pad,), np.uint8)], axis=-1)
        return np.ascontiguousarray(c).view("<i4")

    ca, cb = codes(sa), codes(sb)
    sfa = np.ascontiguousarray(np.swapaxes(pack(np.ascontiguousarray(np.swapaxes(ca, -1, -2))), -1, -2))
    sfb = pack(cb)
    val = lambda c: np.ldexp(1.0, c.astype(np.int32) - 127).astype(np.float32)
    return sfa, sfb, val(ca), val(cb)


def random_ks(num_groups, k_lo, k_hi, seed):
    """K rows per group ~ U{k_lo..k_hi} rounded down to whole 128-wide groups."""
    g = _gen(seed)
    ks = torch.randint(k_lo, k_hi + 1, (num_groups,), generator=g).numpy()
    return (ks // 128 * 128).astype(np.int32)


def masked_problem(num_groups, max_m, N, K, expected_m, seed, m_lo=1):
    """M-grouped masked problem: masked_m[g] ~ U{m_lo..2*expected_m}, capped at
    max_m.  Rows past masked_m[g] of A hold random codes too."""
    g = _gen(seed)
    mm = torch.randint(m_lo, 2 * expected_m + 1, (num_groups,), generator=g).clamp_max(max_m)
    a = torch.randn(num_groups, max_m, K, generator=g, dtype=torch.float32)
    b = torch.randn(num_groups, N, K, generator=g, dtype=torch.float32)
    A, sa = quantize_lhs(a)
    B, sb = quantize_rhs(b)
    return dict(A=A.numpy(), sa=sa.numpy(), B=B.numpy(), sb=sb.numpy(),
                masked_m=mm.numpy().astype(np.int32), G=num_groups, max_m=max_m, N=N, K=K)


def random_codes(shape, seed, lo=0, hi=256, exclude_nan=True):
    """Uniform random e4m3 codes (uint8), NaN codes 0x7F/0xFF replaced by 0."""
    g = _gen(seed)
    c = torch.randint(lo, hi, tuple(shape), generator=g, dtype=torch.int32).to(torch.uint8)
    c = c.numpy()
    if exclude_nan:
        c = np.where((c & 0x7F) == 0x7F, np.uint8(0), c).astype(np.uint8)
    return c


def activation_problem(M, K, seed):
    """A bf16 activation matrix [M,K] (N(0,1), as bit patterns) for the 1x128
    quantiser, and the TMA-aligned leading dimension of its scales."""
    g = _gen(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return dict(X=x.view(torch.int16).numpy().view(np.uint16), M=M, K=K,
                ld_sa=tma_aligned_ld(M))


BF16_SENTINEL = 0xFFFF  # a NaN pattern no computed output can take

#: Named workloads (shapes as the pages' DeepSeek-V3/R1 inference sweep).
CONFIGS = {
    "dense_tiny": dict(kind="dense", cases=[(128, 256, 512)], seed=1000),
    "dense_decode": dict(kind="dense", cases=[(m, n, k) for m in (64, 128) for (n, k) in DENSE_NK],
                         seed=1001),
    "dense_prefill": dict(kind="dense", cases=[(4096, n, k) for (n, k) in DENSE_NK], seed=1002),
    "grouped_contiguous": dict(kind="contiguous", groups=4, m_range=(6144, 10240),
                               nk=GROUPED_NK, seed=1003),
    "grouped_masked": dict(kind="masked", groups=(1, 2, 4, 8), max_m=1024, expected_m=256,
                           nk=GROUPED_NK, seed=1004),
    # MoE weight gradient: per expert dW [M, N] = dY^T X over its tokens (K);
    # (M, N) = (4096, 7168) for the fused gate/up projection, (7168, 2048) for
    # the down projection; tokens per expert ~ U{2048..6144}
    "k_grouped_wgrad": dict(kind="k_grouped", groups=4, k_range=(2048, 6144),
                            mn=[(4096, 7168), (7168, 2048)], seed=1006),
    # the activations feeding the dense sweeps: A [M, K] for every M and K above
    "quantize_act": dict(kind="quantize",
                         cases=[(m, k) for m in (64, 128, 4096) for k in
                                sorted({k for _, k in DENSE_NK})], seed=1005),
}

"""Checks that pin the CPU oracle to something other than itself.

Each `check_*` function takes an `oracle.Oracle` (the normal build, or a
test-only mutant with one planted mistake) and raises AssertionError when the
oracle disagrees with an independent ground truth:

  * the e4m3 and bf16 format definitions (golden fixtures under tests/golden),
  * torch's own float8_e4m3fn -> float64 and float32 -> bfloat16 conversions,
  * a brute-force bf16 rounding that searches the sorted table of all bf16
    values with exact rational arithmetic,
  * exact rational (integer) evaluation of the GEMM written per K element
    (sum_k a*b*sa*sb, no grouping), a different form of the same definition,
  * exact integer results, identity rows, linearity and transposition,
  * a float64 closed form built from torch.matmul on pre-scaled operands,
  * grouped results equal to per-expert / per-group dense runs, with padding
    rows +0 and masked rows untouched, bit for bit.

The GEMM definition these follow: DeepGEMM (es.news.hada.io/topic?id=19459),
"Interfaz GEMM y restricciones de layout" and "Dense y Grouped GEMM".
"""
import bisect
import os
from fractions import Fraction

import numpy as np
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ ground truth --
def torch_e4m3_values():
    """All 256 e4m3 codes decoded by torch (float64)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


_BF16_POS = None


def _bf16_table():
    """Sorted exact values of all finite non-negative bf16 patterns 0x0000..0x7F7F."""
    global _BF16_POS
    if _BF16_POS is None:
        pats = torch.arange(0, 0x7F80, dtype=torch.int32).to(torch.int16)
        _BF16_POS = pats.view(torch.bfloat16).to(torch.float64).tolist()
    return _BF16_POS


def bf16_bruteforce(x):
    """Round x (float or Fraction) to bf16 bits by searching all bf16 values.

    Nearest value wins; at an exact tie the even bit pattern wins; past the
    largest finite value the result is inf when x is at least half a spacing
    beyond it (IEEE roundTiesToEven)."""
    if isinstance(x, float):
        if x != x:
            return 0x7FC0
        if x in (float("inf"), float("-inf")):
            return 0x7F80 if x > 0 else 0xFF80
        neg = np.signbit(x)
        ax = Fraction(abs(x))
    else:
        neg = x < 0
        ax = abs(x)
    tab = _bf16_table()
    top = Fraction(tab[-1])
    half_ulp_top = Fraction(2) ** 119
    if ax >= top + half_ulp_top:
        pat = 0x7F80
    elif ax >= top:
        pat = 0x7F7F
    else:
        i = bisect.bisect_left(tab, float(ax))
        # candidates around ax (float(ax) may be rounded; check neighbours exactly)
        cands = [j for j in (i - 2, i - 1, i, i + 1) if 0 <= j < len(tab)]
        best = None
        for j in cands:
            d = abs(Fraction(tab[j]) - ax)
            key = (d, j & 1)
            if best is None or key < best[0]:
                best = (key, j)
        pat = best[1]
    return pat | (0x8000 if neg else 0)


def e4m3_exact(codes):
    """Exact value of each code as a Fraction (via torch's decode, which is
    exact in float64)."""
    vals = torch_e4m3_values()
    return [Fraction(float(vals[c])) for c in np.asarray(codes).ravel()]


def gemm_exact_bits(A, sa, B, sb):
    """Exact GEMM by rational arithmetic, written per K element:
    D[m,n] = sum_k a[m,k] * b[n,k] * sa[m, k//128] * sb[n//128, k//128],
    then the brute-force bf16 rounding."""
    M, K = A.shape
    N = B.shape[0]
    vals = torch_e4m3_values()
    # every e4m3 value is an integer multiple of 2^-9
    ai = (np.rint(vals[A.astype(np.int64)] * 512)).astype(np.int64)
    bi = (np.rint(vals[B.astype(np.int64)] * 512)).astype(np.int64)
    out = np.zeros((M, N), np.uint16)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for k in range(K):
                p = int(ai[m, k]) * int(bi[n, k])
                if p:
                    tot += Fraction(p, 1 << 18) * Fraction(float(sa[k // 128, m])) \
                        * Fraction(float(sb[n // 128, k // 128]))
            out[m, n] = bf16_bruteforce(tot)
    return out


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _pow2_scales(shape, rng, lo=-3, hi=3):
    return np.ldexp(1.0, rng.integers(lo, hi + 1, size=shape)).astype(np.float32)


# ------------------------------------------------------------------ checks --
def check_e4m3_golden(orc):
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code_s, val_s = line.split()
            got = orc.e4m3_to_double(int(code_s, 16))
            if val_s == "nan":
                assert got != got, (code_s, got)
            else:
                want = float.fromhex(val_s) if "p" in val_s else float(val_s)
                assert got == want and np.signbit(got) == np.signbit(want), (code_s, got, want)


def check_e4m3_all_codes(orc):
    ref = torch_e4m3_values()
    for c in range(256):
        got = orc.e4m3_to_double(c)
        if ref[c] != ref[c]:
            assert got != got, c
        else:
            assert got == ref[c] and np.signbit(got) == np.signbit(ref[c]), (c, got, ref[c])


def check_bf16_golden(orc):
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            x_s, bits_s = line.split()[:2]
            x = float(x_s) if x_s in ("inf", "-inf") else float.fromhex(x_s)
            got = orc.bf16_rne(x)
            assert got == int(bits_s, 16), (x_s, hex(got), bits_s)


def check_bf16_bruteforce(orc, n=4000, seed=7):
    rng = np.random.default_rng(seed)
    # doubles spread over the whole bf16 range, subnormals and overflow included
    exps = rng.integers(-140, 131, size=n)
    mant = rng.random(n) + 1.0
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    xs = sign * np.ldexp(mant, exps)
    # and values sitting exactly on, just above and just below rounding ties
    base = np.ldexp(rng.integers(128, 256, size=n // 4).astype(np.float64) + 0.5,
                    rng.integers(-120, 100, size=n // 4))
    xs = np.concatenate([xs, base, np.nextafter(base, np.inf), np.nextafter(base, -np.inf)])
    for x in xs.tolist():
        got = orc.bf16_rne(x)
        want = bf16_bruteforce(x)
        assert got == want, (x.hex(), hex(got), hex(want))


def check_bf16_vs_torch_float32(orc, n=20000, seed=11):
    """On fp32 inputs torch's fp32 -> bf16 cast is a single RNE rounding."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, w in zip(f.astype(np.float64).tolist(), want.tolist()):
        assert orc.bf16_rne(x) == w, (x, w)


def check_gemm_bruteforce(orc, seed=3):
    """Random codes and random fp32 scales, exact rational ground truth.
    N = 136 crosses a 128-row B scale block; K = 256 has two K groups."""
    for (M, N, K) in ((2, 136, 256), (3, 4, 128), (1, 1, 384)):
        A = W.random_codes((M, K), seed)
        B = W.random_codes((N, K), seed + 1)
        rng = np.random.default_rng(seed)
        sa = np.zeros((K // 128, W.tma_aligned_ld(M)), np.float32)
        sa[:, :M] = rng.uniform(0.01, 2.0, size=(K // 128, M)).astype(np.float32)
        sb = rng.uniform(0.01, 2.0, size=((N + 127) // 128, K // 128)).astype(np.float32)
        got = orc.gemm_nt(A, sa, B, sb)
        want = gemm_exact_bits(A, sa, B, sb)
        assert np.array_equal(got, want), (M, N, K, np.argwhere(got != want)[:5])


# integer-valued e4m3 codes: 0, +-1 .. +-16 (every integer up to 16 is exact in e4m3)
def _int_codes():
    vals = torch_e4m3_values()
    ints = {}
    for c in range(256):
        v = vals[c]
        if v == v and v == int(v) and abs(v) <= 16 and not (v == 0 and c != 0):
            ints[int(v)] = c
    return ints


def check_gemm_exact_integers(orc, seed=5):
    """Integer-valued inputs and power-of-two scales: every partial sum is an
    exact integer times a power of two, so the result is known exactly."""
    ints = _int_codes()
    keys = np.array(sorted(ints))
    rng = np.random.default_rng(seed)
    M, N, K = 9, 200, 512
    av = rng.choice(keys, size=(M, K))
    bv = rng.choice(keys, size=(N, K))
    # sparse copy keeps |D| < 256, where bf16 holds every integer
    av_sp = np.where(rng.random((M, K)) < 0.03, np.clip(av, -2, 2), 0)
    bv_sp = np.where(rng.random((N, K)) < 0.03, np.clip(bv, -2, 2), 0)
    for (a_int, b_int, pow2) in ((av, bv, True), (av_sp, bv_sp, False)):
        A = np.vectorize(ints.get)(a_int).astype(np.uint8)
        B = np.vectorize(ints.get)(b_int).astype(np.uint8)
        kb, nb = K // 128, (N + 127) // 128
        if pow2:
            sa = np.zeros((kb, W.tma_aligned_ld(M)), np.float32)
            sa[:, :M] = _pow2_scales((kb, M), rng)
            sb = _pow2_scales((nb, kb), rng)
        else:
            sa = np.ones((kb, W.tma_aligned_ld(M)), np.float32)
            sb = np.ones((nb, kb), np.float32)
        got = orc.gemm_nt(A, sa, B, sb)
        want = np.zeros((M, N), np.uint16)
        for m in range(M):
            for n in range(N):
                tot = Fraction(0)
                for g in range(kb):
                    d = int(np.dot(a_int[m, 128 * g:128 * g + 128].astype(np.int64),
                                   b_int[n, 128 * g:128 * g + 128].astype(np.int64)))
                    tot += d * Fraction(float(sa[g, m])) * Fraction(float(sb[n // 128, g]))
                want[m, n] = bf16_bruteforce(tot)
                if not pow2:
                    assert abs(tot) < 256 and tot.denominator == 1
        assert np.array_equal(got, want), np.argwhere(got != want)[:5]


def check_gemm_identity(orc, seed=9):
    """Row m of A is one-hot 1.0 at column k0 with sa = 1, so row m of D is
    B[:, k0] * sb[n//128, k0//128] rounded once to bf16."""
    M, N, K = 4, 260, 384
    B = W.random_codes((N, K), seed)
    rng = np.random.default_rng(seed)
    sb = rng.uniform(0.01, 4.0, size=((N + 127) // 128, K // 128)).astype(np.float32)
    A = np.zeros((M, K), np.uint8)
    k0s = [0, 129, 255, 383]
    for m, k0 in enumerate(k0s):
        A[m, k0] = 0x38  # 1.0
    sa = np.ones((K // 128, W.tma_aligned_ld(M)), np.float32)
    got = orc.gemm_nt(A, sa, B, sb)
    vals = torch_e4m3_values()
    for m, k0 in enumerate(k0s):
        for n in range(N):
            exact = Fraction(float(vals[B[n, k0]])) * Fraction(float(sb[n // 128, k0 // 128]))
            assert got[m, n] == bf16_bruteforce(exact), (m, n)


def check_gemm_linearity_transpose(orc, seed=13):
    rng = np.random.default_rng(seed)
    M, N, K = 6, 300, 384
    A = W.random_codes((M, K), seed)
    B = W.random_codes((N, K), seed + 1)
    kb, nb = K // 128, (N + 127) // 128
    sa = np.zeros((kb, W.tma_aligned_ld(M)), np.float32)
    sa[:, :M] = rng.uniform(0.5, 2.0, size=(kb, M)).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, size=(nb, kb)).astype(np.float32)
    D0 = _f(orc.gemm_nt(A, sa, B, sb))
    # all groups of row 2 scaled by 2^3 -> row 2 scaled by 2^3 exactly
    sa2 = sa.copy(); sa2[:, 2] *= 8.0
    D1 = _f(orc.gemm_nt(A, sa2, B, sb))
    exp = D0.copy(); exp[2] *= 8.0
    assert np.array_equal(D1, exp)
    # all groups of B block 1 scaled by 2^-2 -> columns 128..255 scaled by 2^-2
    sb2 = sb.copy(); sb2[1, :] *= 0.25
    D2 = _f(orc.gemm_nt(A, sa, B, sb2))
    exp = D0.copy(); exp[:, 128:256] *= 0.25
    assert np.array_equal(D2, exp)
    # one K group's scales zeroed -> equals the GEMM on that group's zeroed codes
    sa3 = sa.copy(); sa3[1, :] = 0.0
    A3 = A.copy(); A3[:, 128:256] = 0
    assert np.array_equal(orc.gemm_nt(A, sa3, B, sb), orc.gemm_nt(A3, sa, B, sb))
    # transposition: with 128x128 blocks on both sides and per-group constant
    # scales, swapping the operands (and their scales) transposes D
    Mt = Nt = 128
    At = W.random_codes((Mt, K), seed + 2)
    Bt = W.random_codes((Nt, K), seed + 3)
    alpha = rng.uniform(0.5, 2.0, size=kb).astype(np.float32)
    beta = rng.uniform(0.5, 2.0, size=kb).astype(np.float32)
    sa_t = np.repeat(alpha[:, None], Mt, axis=1)
    sb_t = beta[None, :].copy()
    sa_s = np.repeat(beta[:, None], Nt, axis=1)
    sb_s = alpha[None, :].copy()
    D = orc.gemm_nt(At, sa_t, Bt, sb_t)
    Ds = orc.gemm_nt(Bt, sa_s, At, sb_s)
    assert np.array_equal(D, Ds.T)


def check_gemm_closed_form(orc, seed=17):
    """float64 torch.matmul on decoded, pre-scaled operands equals the
    oracle's unrounded accumulators to ~1e-13 relative."""
    M, N, K = 33, 257, 640
    p = W.dense_problem(M, N, K, seed)
    vals = torch.from_numpy(torch_e4m3_values())
    Ad = vals[torch.from_numpy(p["A"]).long()]
    Bd = vals[torch.from_numpy(p["B"]).long()]
    sa_exp = torch.from_numpy(p["sa"][:, :M]).double().T.repeat_interleave(128, dim=1)
    sb_exp = torch.from_numpy(p["sb"]).double().repeat_interleave(128, dim=0)[:N] \
        .repeat_interleave(128, dim=1)
    ref = ((Ad * sa_exp) @ (Bd * sb_exp).T).numpy()
    mag = (torch.abs(Ad * sa_exp) @ torch.abs(Bd * sb_exp).T).numpy()
    acc = orc.gemm_nt_f64(p["A"], p["sa"], p["B"], p["sb"])
    assert np.all(np.abs(acc - ref) <= 1e-13 * mag + 1e-300)
    bits = orc.gemm_nt(p["A"], p["sa"], p["B"], p["sb"])
    assert np.array_equal(bits, np.vectorize(bf16_bruteforce, otypes=[np.uint16])(acc))


def check_grouped_contiguous(orc, seed=19):
    p = W.contiguous_problem(3, 136, 256, 1, 200, seed)
    D = orc.grouped_contiguous(p["A"], p["sa"], p["B"], p["sb"], p["m_indices"])
    mi = p["m_indices"]
    assert np.all(D[mi < 0] == 0)  # +0 bit pattern on padding rows
    assert (mi < 0).any()
    for e in range(p["G"]):
        rows = np.nonzero(mi == e)[0]
        dense = orc.gemm_nt_rows(p["A"], p["sa"], p["B"][e], p["sb"][e], rows)
        assert np.array_equal(D[rows], dense), e
    # a row subset gives the same rows
    sub = np.array([0, 5, len(mi) - 1, 130], np.int64)
    assert np.array_equal(orc.grouped_contiguous(p["A"], p["sa"], p["B"], p["sb"], mi, rows=sub),
                          D[sub])


def check_grouped_masked(orc, seed=23):
    p = W.masked_problem(3, 200, 136, 256, 60, seed)
    G, max_m, N = p["G"], p["max_m"], p["N"]
    init = np.full((G, max_m, N), W.BF16_SENTINEL, np.uint16)
    D = orc.grouped_masked(p["A"], p["sa"], p["B"], p["sb"], p["masked_m"], init)
    for g in range(G):
        v = int(p["masked_m"][g])
        assert np.all(D[g, v:] == W.BF16_SENTINEL)
        dense = orc.gemm_nt(p["A"][g], p["sa"][g], p["B"][g], p["sb"][g])
        assert np.array_equal(D[g, :v], dense[:v]), g
    assert (p["masked_m"] < max_m).all()


# --------------------------------------------------- D = C + A @ B^T -----
def check_gemm_with_c(orc, seed=37):
    """The addend form against independent results: C = 0 gives the plain
    product; all-zero A gives C back bit for bit; integer-valued C (|C| < 64)
    plus a sparse integer GEMM (|sum| < 64, unit scales) gives the exact
    integer C + sum, which bf16 holds."""
    ints = _int_codes()
    rng = np.random.default_rng(seed)
    p = W.dense_problem(7, 136, 384, seed)
    zero = np.zeros((7, 136), np.uint16)
    assert np.array_equal(orc.gemm_nt_c(p["A"], p["sa"], p["B"], p["sb"], zero),
                          orc.gemm_nt(p["A"], p["sa"], p["B"], p["sb"]))
    C = torch.from_numpy(rng.standard_normal((7, 136)).astype(np.float32)).to(torch.bfloat16)
    Cb = C.view(torch.int16).numpy().view(np.uint16)
    A0 = np.zeros_like(p["A"])
    assert np.array_equal(orc.gemm_nt_c(A0, p["sa"], p["B"], p["sb"], Cb), Cb)
    M, N, K = 6, 140, 256
    av = np.where(rng.random((M, K)) < 0.03, rng.integers(-2, 3, (M, K)), 0)
    bv = np.where(rng.random((N, K)) < 0.03, rng.integers(-2, 3, (N, K)), 0)
    A = np.vectorize(ints.get)(av).astype(np.uint8)
    B = np.vectorize(ints.get)(bv).astype(np.uint8)
    sa = np.ones((K // 128, W.tma_aligned_ld(M)), np.float32)
    sb = np.ones(((N + 127) // 128, K // 128), np.float32)
    c_int = rng.integers(-40, 41, (M, N))
    Cb = torch.from_numpy(c_int.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    exact = c_int + av.astype(np.int64) @ bv.astype(np.int64).T
    assert np.abs(exact).max() < 256
    want = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.gemm_nt_c(A, sa, B, sb, Cb), want)


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def check_gemm_layouts(orc, seed=41):
    """nn / tn / tt against gemm_nt on the same logical operands, transposed
    here by numpy (M, N, K all different and N ragged, so a swapped or
    transposed index cannot pass); "nt" through the layout routine equals
    gemm_nt; the addend enters as in gemm_nt_c."""
    p = W.dense_problem(40, 136, 384, seed)
    A, B, sa, sb = p["A"], p["B"], p["sa"], p["sb"]
    At, Bt = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)   # [K, M], [K, N]
    want = orc.gemm_nt(A, sa, B, sb)
    stored = {"nt": (A, B), "nn": (A, Bt), "tn": (At, Bt), "tt": (At, B)}
    for layout, (a, b) in stored.items():
        got = orc.gemm_layout(layout, a, sa, b, sb)
        assert np.array_equal(got, want), f"layout {layout}"
    rng = np.random.default_rng(seed)
    C = _bf16_bits(rng.standard_normal((40, 136)))
    assert np.array_equal(orc.gemm_layout("tn", At, sa, Bt, sb, C), orc.gemm_nt_c(A, sa, B, sb, C))


def check_k_grouped(orc, seed=43):
    """K-grouped tn: each group equals gemm_nt_c on its own K slice (operands
    transposed by numpy, the slice's scale rows and columns), an empty group
    returns C (or +0) bit for bit, and one group over all of K equals the tn
    layout."""
    rng = np.random.default_rng(seed)
    M, N = 40, 136
    ks = np.array([256, 0, 384, 128], np.int32)
    K_all = int(ks.sum())
    kb = K_all // 128
    A = W.random_codes((K_all, M), seed + 1)             # [K_all, M]
    B = W.random_codes((K_all, N), seed + 2)             # [K_all, N]
    sa = (rng.random((kb, W.tma_aligned_ld(M))) + 0.25).astype(np.float32)
    sb = (rng.random(((N + 127) // 128, kb)) + 0.25).astype(np.float32)
    C = _bf16_bits(rng.standard_normal((len(ks), M, N)))
    D = orc.k_grouped_tn(A, sa, B, sb, ks, C)
    D0 = orc.k_grouped_tn(A, sa, B, sb, ks)
    k0 = 0
    for g, kg in enumerate(ks):
        if kg == 0:
            assert np.array_equal(D[g], C[g]), f"empty group {g} must return C"
            assert not np.any(D0[g]), f"empty group {g} without C must be +0"
            continue
        j0, j1 = k0 // 128, (k0 + kg) // 128
        Ag = np.ascontiguousarray(A[k0:k0 + kg].T)
        Bg = np.ascontiguousarray(B[k0:k0 + kg].T)
        sag = np.ascontiguousarray(sa[j0:j1])
        sbg = np.ascontiguousarray(sb[:, j0:j1])
        assert np.array_equal(D[g], orc.gemm_nt_c(Ag, sag, Bg, sbg, C[g])), f"group {g}"
        assert np.array_equal(D0[g], orc.gemm_nt(Ag, sag, Bg, sbg)), f"group {g} without C"
        k0 += kg
    one = orc.k_grouped_tn(A, sa, B, sb, np.array([K_all], np.int32))
    assert np.array_equal(one[0], orc.gemm_layout("tn", A, sa, B, sb))


# ------------------------------------------------- activation quantiser --
def _torch_e4m3_bits(v):
    """torch's float32 -> float8_e4m3fn cast of v clamped to +-448 (its cast
    does not saturate), as code bytes."""
    t = torch.from_numpy(np.asarray(v, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def check_e4m3_encode_vs_torch(orc, seed=29):
    """The oracle's fp32 -> e4m3 rounding against torch's on every code value,
    every midpoint between neighbouring values (the ties), values past the
    largest finite one, the subnormal range and random magnitudes."""
    vals = torch_e4m3_values()
    fin = np.unique(vals[np.isfinite(vals)])
    mids = (fin[:-1] + fin[1:]) / 2                  # exact in fp32
    rng = np.random.default_rng(seed)
    rnd = rng.standard_normal(3000) * np.exp2(rng.integers(-14, 10, 3000))
    extra = [448.0, 449.0, 463.9, 464.0, 465.0, 1e6, -1e6, 2.0 ** -6, 2.0 ** -9, 2.0 ** -10,
             3 * 2.0 ** -10, -(2.0 ** -10), 0.0, -0.0]
    v = np.concatenate([fin, mids, rnd, extra]).astype(np.float32)
    want = _torch_e4m3_bits(v)
    got = np.array([orc.e4m3_from_float(x) for x in v], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (v[bad[:5]], got[bad[:5]], want[bad[:5]])


def check_quantize_invariants(orc, seed=31):
    """Properties any correct 1x128 quantiser of this reading has, checked per
    (row, group) on bf16 inputs spread over 40 binades: scale * 448 recovers
    max(amax, 1e-4); the group maximum maps to code magnitude 448; every code
    is x / scale rounded to the nearest e4m3 value (within half a step, signs
    kept); zero and below-floor groups; scale columns past M untouched."""
    rng = np.random.default_rng(seed)
    G, M, K = 2, 5, 512
    x = rng.standard_normal((G, M, K))
    x *= np.repeat(np.exp2(rng.integers(-20, 20, (G, M, K // 128))), 128, axis=-1)
    x[0, 1, 128:256] = 0.0                        # an all-zero group
    x[1, 2, :128] = 1e-6 * np.sign(x[1, 2, :128])   # below the 1e-4 floor
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xf = xb.to(torch.float64).numpy()            # the exact bf16 values
    Q, sa = orc.quantize_1x128(bits, ld_sa=8)
    assert Q.shape == (G, M, K) and sa.shape == (G, K // 128, 8)
    assert np.all(np.isnan(sa[:, :, M:])), "scale columns past M written"
    dec = torch_e4m3_values()[Q.astype(np.int64)]
    for z in range(G):
        for m in range(M):
            for g in range(K // 128):
                blk = xf[z, m, g * 128:(g + 1) * 128]
                d = dec[z, m, g * 128:(g + 1) * 128]
                s = float(sa[z, g, m])
                amax = float(np.abs(blk).max())
                a = max(amax, 1e-4)
                assert abs(s * 448.0 - a) <= a * 2.0 ** -22, (z, m, g, s, amax)
                if amax > 1e-4:
                    assert np.abs(d).max() == 448.0, (z, m, g)
                t = np.clip(blk / s, -448.0, 448.0)
                half = np.maximum(np.abs(t) * 2.0 ** -4, 2.0 ** -10) * (1 + 2.0 ** -20)
                assert np.all(np.abs(d - t) <= half), (z, m, g)
                assert np.all(d * t >= 0), (z, m, g)   # no sign flips
    assert np.all(Q[0, 1, 128:256] & 0x7F == 0)


# ------------------------------------------------- UE8M0 packed scales --
def _pack_ue8m0(codes):
    """uint8 exponent codes [..., n] -> int32 words [..., ceil(n/4)], four
    consecutive codes per word, the first in the lowest byte: a numpy byte
    view (little-endian), independent of the oracle's shifts."""
    codes = np.asarray(codes, np.uint8)
    n = codes.shape[-1]
    pad = (-n) % 4
    if pad:
        codes = np.concatenate([codes, np.zeros(codes.shape[:-1] + (pad,), np.uint8)], axis=-1)
    return np.ascontiguousarray(codes).view("<i4")


def check_ue8m0_codes(orc):
    """All 256 UE8M0 codes: 2^(e - 127) (numpy's ldexp), 0xFF NaN; and the
    format's worked values."""
    for e in range(255):
        assert orc.ue8m0_to_double(e) == float(np.ldexp(1.0, e - 127)), e
    assert np.isnan(orc.ue8m0_to_double(255))
    assert orc.ue8m0_to_double(0x7F) == 1.0 and orc.ue8m0_to_double(0x80) == 2.0
    assert orc.ue8m0_to_double(0x7E) == 0.5 and orc.ue8m0_to_double(0) == 2.0 ** -127


def check_ue8m0_packing(orc, seed=47):
    """Scales packed by a numpy byte view decode back to themselves, for
    K group counts that do and do not fill the last word."""
    rng = np.random.default_rng(seed)
    for kb in (1, 4, 5, 7, 9):
        ld, nb = 12, 3
        ea = rng.integers(100, 150, (kb, ld)).astype(np.uint8)      # [kb, ld] codes
        eb = rng.integers(100, 150, (nb, kb)).astype(np.uint8)      # [nb, kb]
        sfa = np.ascontiguousarray(_pack_ue8m0(ea.T).T)             # [ceil(kb/4), ld]
        sfb = _pack_ue8m0(eb)                                       # [nb, ceil(kb/4)]
        assert np.array_equal(orc.decode_sfa(sfa, kb), np.ldexp(1.0, ea.astype(int) - 127)), kb
        assert np.array_equal(orc.decode_sfb(sfb, kb), np.ldexp(1.0, eb.astype(int) - 127)), kb


def check_gemm_ue8m0(orc, seed=53):
    """The packed-scale GEMM equals gemm_nt with the same scales given in
    fp32, and gives exact integers for integer operands with power-of-two
    scales whose products cancel."""
    rng = np.random.default_rng(seed)
    p = W.dense_problem(9, 200, 640, seed)
    kb = 5
    ea = rng.integers(120, 134, (kb, 12)).astype(np.uint8)
    eb = rng.integers(120, 134, (2, kb)).astype(np.uint8)
    sfa = np.ascontiguousarray(_pack_ue8m0(ea.T).T)
    sfb = _pack_ue8m0(eb)
    sa = np.ldexp(1.0, ea.astype(int) - 127).astype(np.float32)
    sb = np.ldexp(1.0, eb.astype(int) - 127).astype(np.float32)
    assert np.array_equal(orc.gemm_nt_ue8m0(p["A"], sfa, p["B"], sfb),
                          orc.gemm_nt(p["A"], sa, p["B"], sb))
    ints = _int_codes()
    M, N, K = 4, 130, 512
    av = np.where(rng.random((M, K)) < 0.05, rng.integers(-2, 3, (M, K)), 0)
    bv = np.where(rng.random((N, K)) < 0.05, rng.integers(-2, 3, (N, K)), 0)
    A = np.vectorize(ints.get)(av).astype(np.uint8)
    B = np.vectorize(ints.get)(bv).astype(np.uint8)
    # sa = 2^+k, sb = 2^-k per group: every product of scales is 1
    k = rng.integers(-5, 6, K // 128)
    ea = np.repeat((127 + k)[:, None], 4, axis=1).astype(np.uint8)          # [kb, 4]
    eb = np.repeat((127 - k)[None, :], 2, axis=0).astype(np.uint8)          # [2, kb]
    sfa = np.ascontiguousarray(_pack_ue8m0(ea.T).T)
    sfb = _pack_ue8m0(eb)
    exact = av.astype(np.int64) @ bv.astype(np.int64).T
    want = _bf16_bits(exact.astype(np.float32))
    assert np.array_equal(orc.gemm_nt_ue8m0(A, sfa, B, sfb), want)


def check_quantize_ue8m0(orc, seed=59):
    """The UE8M0 quantiser: every scale a power of two s, the smallest one
    >= fp32(max(amax, 1e-4) / 448) (s / 2 is below it), codes x / s rounded to
    the nearest e4m3 (within half a step, signs kept), zero and below-floor
    groups; bytes of groups past K/128 untouched."""
    rng = np.random.default_rng(seed)
    G, M, K = 2, 5, 640                        # 5 K groups: the second word half used
    x = rng.standard_normal((G, M, K))
    x *= np.repeat(np.exp2(rng.integers(-20, 20, (G, M, K // 128))), 128, axis=-1)
    x[0, 1, 128:256] = 0.0
    x[1, 2, :128] = 1e-6 * np.sign(x[1, 2, :128])
    x[0, 3, :128] = 448.0 * 2.0 ** 5 * np.sign(x[0, 3, :128]) * (np.arange(128) / 127.0)
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xf = xb.to(torch.float64).numpy()
    fill = np.int32(0x5A5A5A5A)
    Q, sfa = orc.quantize_1x128_ue8m0(bits, ld=8, fill=fill)
    assert sfa.shape == (G, 2, 8)
    raw = np.ascontiguousarray(sfa).view(np.uint8).reshape(G, 2, 8, 4)
    assert np.all(raw[:, 1, :, 1:] == 0x5A), "bytes past K/128 written"
    assert np.all(sfa[:, :, M:] == fill), "columns past M written"
    dec = torch_e4m3_values()[Q.astype(np.int64)]
    for z in range(G):
        for m in range(M):
            for g in range(K // 128):
                e = int(raw[z, g // 4, m, g % 4])
                s = float(np.ldexp(1.0, e - 127))
                blk = xf[z, m, g * 128:(g + 1) * 128]
                a = np.float32(max(float(np.abs(blk).max()), 1e-4))
                t = float(np.float32(a) / np.float32(448.0))
                assert s >= t and s / 2 < t, (z, m, g, s, t)
                u = np.clip(blk / s, -448.0, 448.0)
                half = np.maximum(np.abs(u) * 2.0 ** -4, 2.0 ** -10) * (1 + 2.0 ** -20)
                d = dec[z, m, g * 128:(g + 1) * 128]
                assert np.all(np.abs(d - u) <= half), (z, m, g)
                assert np.all(d * u >= 0), (z, m, g)
    assert raw[0, 0, 3, 0] == 127 + 5     # amax = 448 * 2^5 exactly: s = 2^5


ALL_CHECKS = [
    check_gemm_layouts, check_k_grouped, check_ue8m0_codes, check_ue8m0_packing,
    check_gemm_ue8m0, check_quantize_ue8m0,
    check_e4m3_golden, check_e4m3_all_codes, check_bf16_golden, check_bf16_bruteforce,
    check_bf16_vs_torch_float32, check_gemm_bruteforce, check_gemm_exact_integers,
    check_gemm_identity, check_gemm_linearity_transpose, check_gemm_closed_form,
    check_grouped_contiguous, check_grouped_masked, check_e4m3_encode_vs_torch,
    check_quantize_invariants, check_gemm_with_c,
]

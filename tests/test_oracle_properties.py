"""Randomised checks of the CPU oracle against independent ground truth (no GPU):
exact rational arithmetic for the dense and K-grouped forms on tiny random
problems, the layout forms against numpy-transposed operands, and the packed
UE8M0 scales against a numpy byte view.  Hypothesis draws the shapes and a seed;
the codes and scales come from numpy with that seed; each example is small
enough for Fraction arithmetic."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from tests import oracle_checks as C  # noqa: E402

ORC = oracle.Oracle()
SETTINGS = settings(max_examples=12, deadline=None, derandomize=True)

# every e4m3 code except the two NaN patterns
CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)


def _codes(rng, shape):
    return rng.choice(CODES, size=shape).astype(np.uint8)


def _scales(rng, shape):
    """fp32 scales of random mantissa and exponent in [2^-8, 2^8)."""
    mant = rng.uniform(1.0, 2.0, size=shape).astype(np.float32)
    return np.ldexp(mant, rng.integers(-8, 8, size=shape)).astype(np.float32)


@st.composite
def dense_problems(draw):
    M = draw(st.integers(1, 3))
    N = draw(st.sampled_from([1, 2, 5, 129]))
    K = 128 if N > 5 else draw(st.sampled_from([128, 256]))
    if N > 5:
        M = 1
    rng = np.random.default_rng(draw(st.integers(0, 2**31 - 1)))
    A = _codes(rng, (M, K))
    B = _codes(rng, (N, K))
    ld = (M + 3) // 4 * 4
    sa = np.zeros((K // 128, ld), np.float32)
    sa[:, :M] = _scales(rng, (K // 128, M))
    sb = _scales(rng, ((N + 127) // 128, K // 128))
    return A, sa, B, sb


@SETTINGS
@given(dense_problems())
def test_gemm_nt_equals_exact_rational(prob):
    A, sa, B, sb = prob
    assert np.array_equal(ORC.gemm_nt(A, sa, B, sb), C.gemm_exact_bits(A, sa, B, sb))


@SETTINGS
@given(dense_problems(), st.sampled_from(["nn", "tn", "tt"]))
def test_layouts_equal_nt(prob, layout):
    A, sa, B, sb = prob
    a = np.ascontiguousarray(A.T) if layout[0] == "t" else A
    b = np.ascontiguousarray(B.T) if layout[1] == "n" else B
    assert np.array_equal(ORC.gemm_layout(layout, a, sa, b, sb), ORC.gemm_nt(A, sa, B, sb))


@st.composite
def k_grouped_problems(draw):
    ks = np.array(draw(st.lists(st.sampled_from([0, 128, 256]), min_size=1, max_size=3)), np.int32)
    if ks.sum() == 0:
        ks[0] = 128
    M = draw(st.integers(1, 2))
    N = draw(st.sampled_from([1, 3, 130]))
    if N > 3:
        M = 1
        ks = np.minimum(ks, 128)
        if ks.sum() == 0:
            ks[0] = 128
    K = int(ks.sum())
    rng = np.random.default_rng(draw(st.integers(0, 2**31 - 1)))
    A = _codes(rng, (K, M))
    B = _codes(rng, (K, N))
    ld = (M + 3) // 4 * 4
    sa = np.zeros((K // 128, ld), np.float32)
    sa[:, :M] = _scales(rng, (K // 128, M))
    sb = _scales(rng, ((N + 127) // 128, K // 128))
    return A, sa, B, sb, ks


@SETTINGS
@given(k_grouped_problems())
def test_k_grouped_equals_exact_rational_per_group(prob):
    A, sa, B, sb, ks = prob
    D = ORC.k_grouped_tn(A, sa, B, sb, ks)
    k0 = 0
    for g, kg in enumerate(ks):
        if kg == 0:
            assert not np.any(D[g])
            continue
        j0, j1 = k0 // 128, (k0 + kg) // 128
        want = C.gemm_exact_bits(np.ascontiguousarray(A[k0:k0 + kg].T),
                                 np.ascontiguousarray(sa[j0:j1]),
                                 np.ascontiguousarray(B[k0:k0 + kg].T),
                                 np.ascontiguousarray(sb[:, j0:j1]))
        assert np.array_equal(D[g], want), g
        k0 += kg


@SETTINGS
@given(st.integers(1, 9), st.integers(1, 6), st.integers(0, 2**31 - 1))
def test_ue8m0_packing_round_trip(kb, ld, seed):
    ea = np.random.default_rng(seed).integers(0, 255, size=(ld, kb)).astype(np.uint8)
    sfa = np.ascontiguousarray(C._pack_ue8m0(ea).T)            # [ceil(kb/4), ld]
    want = np.ldexp(1.0, ea.T.astype(np.int32) - 127)
    assert np.array_equal(ORC.decode_sfa(sfa, kb), want)

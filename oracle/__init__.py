"""CPU oracle for the FP8 fine-grained-scaled GEMM (NT layout, bf16 output).

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` may import this package.  It shares no code with
the CUDA path and never imports it; the two meet only through the seeded inputs
of `workloads`.

The arithmetic lives in `ref_gemm.c` (plain C, double precision, one bf16
rounding at the end); this module loads it with ctypes and marshals numpy
arrays.  See `ref_gemm.c` for the formula and the pages it follows
(DeepGEMM, es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de
layout" and "Dense y Grouped GEMM").

Every function takes and returns numpy arrays:
  A, B          uint8 e4m3 codes, row-major ([M,K] / [N,K], grouped [G,...,K])
  sa            float32, K-group-major: [kb, ld_sa] (masked: [G, kb, ld_sa])
  sb            float32, [nb, kb] (grouped: [G, nb, kb])
  D (returned)  uint16 bf16 bit patterns

Parity status of each function (what pins it, in tests/test_oracle_pins.py):
  e4m3_to_double   pinned: all 256 codes vs the format definition and torch
  bf16_rne         pinned: brute-force neighbour search, constructed ties,
                   double-rounding traps, torch's fp32->bf16 on fp32 inputs
  gemm_nt          pinned: exact rational brute force, exact integer results,
                   identity, linearity/transpose, float64 library closed form
  grouped_*        pinned: equal to per-expert / per-group dense runs,
                   padding rows +0 and masked rows untouched (bit-exact)
  gemm_nt_c        pinned: C = 0 gives gemm_nt; zero A gives C back bit for
                   bit; integer-valued C plus an exact integer GEMM gives the
                   exact integer sum
  gemm_layout      pinned: each of nn / tn / tt equals gemm_nt on the
                   operands transposed by numpy (non-square, ragged N, so a
                   swapped index fails); "nt" through it equals gemm_nt; C
                   handled as in gemm_nt_c
  k_grouped_tn     pinned: every group equals gemm_nt (or gemm_nt_c) on its
                   own K slice transposed by numpy, with its own scale
                   columns; an empty group gives C (or +0) bit for bit; one
                   group over all of K equals gemm_layout "tn"
  ue8m0_to_double  pinned: all 256 codes against 2^(e-127) by ldexp and the
                   format's worked values (0x7F = 1, 0xFF = NaN)
  decode_sfa/sfb   pinned: scales packed here by a numpy byte view (little-
                   endian uint8 [..., 4] as int32) decode back to themselves
  gemm_nt_ue8m0    pinned: equal to gemm_nt with the decoded scales; exact
                   integer results with power-of-two scales
  quantize_1x128_ue8m0  pinned: every scale a power of two, the smallest one
                   >= fp32(amax/448) (tight: half of it is below), codes
                   within half an e4m3 step of x / s, zero groups
  e4m3_from_float  pinned: torch's float32 -> float8_e4m3fn cast (after
                   clamping to +-448) on every code value, every midpoint
                   between neighbours (ties), saturation and random values
  quantize_1x128   pinned: the group maximum maps to code magnitude 448, the
                   scale times 448 recovers the maximum, every code decodes
                   to x / scale within half an e4m3 step, zero groups, layout
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIBS = {}

_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_int = ctypes.c_int


def _load(path):
    lib = ctypes.CDLL(path)
    lib.dg_ref_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.dg_ref_e4m3_to_double.restype = ctypes.c_double
    lib.dg_ref_bf16_rne.argtypes = [ctypes.c_double]
    lib.dg_ref_bf16_rne.restype = ctypes.c_uint16
    lib.dg_ref_max_threads.argtypes = []
    lib.dg_ref_max_threads.restype = _int
    lib.dg_ref_gemm_nt_f64.argtypes = [_u8p, _f32p, _int, _u8p, _f32p, _f64p, _int, _int, _int, _int]
    lib.dg_ref_gemm_nt.argtypes = [_u8p, _f32p, _int, _u8p, _f32p, _u16p, _int, _int, _int, _int]
    lib.dg_ref_gemm_nt_rows.argtypes = [_u8p, _f32p, _int, _u8p, _f32p, _u16p, _int, _int,
                                        _i64p, _int, _int]
    lib.dg_ref_grouped_contiguous_rows.argtypes = [_u8p, _f32p, _int, _u8p, _f32p, _i32p,
                                                   _u16p, _int, _int, _int, _i64p, _int, _int]
    lib.dg_ref_grouped_masked.argtypes = [_u8p, _f32p, _int, _u8p, _f32p, _i32p, _u16p,
                                          _int, _int, _int, _int, _int]
    lib.dg_ref_gemm_nt_c.argtypes = [_u8p, _f32p, _int, _u8p, _f32p, _u16p, _u16p, _int, _int,
                                     _int, _int]
    lib.dg_ref_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.dg_ref_e4m3_from_float.restype = ctypes.c_uint8
    lib.dg_ref_gemm_layout.argtypes = [_u8p, _int, _f32p, _int, _u8p, _int, _f32p, _u16p, _u16p,
                                       _int, _int, _int, _int]
    lib.dg_ref_k_grouped_tn.argtypes = [_u8p, _f32p, _int, _u8p, _f32p, _u16p, _u16p, _int, _int,
                                        _i32p, _int, _int]
    lib.dg_ref_ue8m0_to_double.argtypes = [ctypes.c_uint8]
    lib.dg_ref_ue8m0_to_double.restype = ctypes.c_double
    lib.dg_ref_decode_sfa.argtypes = [_i32p, _f32p, _int, _int]
    lib.dg_ref_decode_sfb.argtypes = [_i32p, _f32p, _int, _int]
    lib.dg_ref_quantize_1x128_ue8m0.argtypes = [_u16p, _u8p, _i32p, _int, _int, _int, _int, _int]
    lib.dg_ref_quantize_1x128.argtypes = [_u16p, _u8p, _f32p, _int, _int, _int, _int, _int]
    for f in ("dg_ref_gemm_nt_f64", "dg_ref_gemm_nt", "dg_ref_gemm_nt_rows",
              "dg_ref_grouped_contiguous_rows", "dg_ref_grouped_masked",
              "dg_ref_quantize_1x128", "dg_ref_gemm_nt_c"):
        getattr(lib, f).restype = None
    return lib


def lib(path=None):
    """The oracle library (built on first use); `path` selects another build
    of the same source (the test-only mutants)."""
    if path is None:
        path = _build.build()
    if path not in _LIBS:
        _LIBS[path] = _load(path)
    return _LIBS[path]


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a, ptype):
    return a.ctypes.data_as(ptype)


class Oracle:
    """Bound view of one oracle build (the normal one unless `path` is given)."""

    def __init__(self, path=None):
        self.lib = lib(path)

    # -- scalar pieces ----------------------------------------------------
    def e4m3_to_double(self, code):
        return self.lib.dg_ref_e4m3_to_double(int(code) & 0xFF)

    def bf16_rne(self, x):
        return int(self.lib.dg_ref_bf16_rne(float(x)))

    def e4m3_from_float(self, v):
        return int(self.lib.dg_ref_e4m3_from_float(float(np.float32(v))))

    def ue8m0_to_double(self, code):
        return self.lib.dg_ref_ue8m0_to_double(int(code) & 0xFF)

    def max_threads(self):
        return int(self.lib.dg_ref_max_threads())

    # -- dense ------------------------------------------------------------
    def gemm_nt_f64(self, A, sa, B, sb, nthreads=0):
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32)
        M, K = A.shape
        N = B.shape[0]
        acc = np.zeros((M, N), np.float64)
        self.lib.dg_ref_gemm_nt_f64(_p(A, _u8p), _p(sa, _f32p), sa.shape[-1], _p(B, _u8p),
                                    _p(sb, _f32p), _p(acc, _f64p), M, N, K, nthreads)
        return acc

    def gemm_nt(self, A, sa, B, sb, nthreads=0):
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32)
        M, K = A.shape
        N = B.shape[0]
        _check_dense(A, sa, B, sb)
        D = np.zeros((M, N), np.uint16)
        self.lib.dg_ref_gemm_nt(_p(A, _u8p), _p(sa, _f32p), sa.shape[-1], _p(B, _u8p),
                                _p(sb, _f32p), _p(D, _u16p), M, N, K, nthreads)
        return D

    def gemm_nt_c(self, A, sa, B, sb, C, nthreads=0):
        """D = bf16(C + sum_g ...): C bf16 bit patterns [M, N]."""
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32); C = _c(C, np.uint16)
        M, K = A.shape
        N = B.shape[0]
        _check_dense(A, sa, B, sb)
        assert C.shape == (M, N)
        D = np.zeros((M, N), np.uint16)
        self.lib.dg_ref_gemm_nt_c(_p(A, _u8p), _p(sa, _f32p), sa.shape[-1], _p(B, _u8p),
                                  _p(sb, _f32p), _p(C, _u16p), _p(D, _u16p), M, N, K, nthreads)
        return D

    def gemm_layout(self, layout, A, sa, B, sb, C=None, nthreads=0):
        """D = bf16(C + A @ B) in storage layout `layout` ("nt", "nn", "tn" or
        "tt"): A [M,K] for "n" or [K,M] for "t"; B [N,K] for "t" or [K,N] for
        "n"; sa [kb, ld_sa]; sb [nb, kb]; C bf16 bits [M, N] or None."""
        assert layout in ("nt", "nn", "tn", "tt")
        a_t, b_n = layout[0] == "t", layout[1] == "n"
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32)
        K, M = A.shape if a_t else A.shape[::-1]
        N = B.shape[1] if b_n else B.shape[0]
        assert (B.shape[0] if b_n else B.shape[1]) == K and K % 128 == 0
        assert sa.ndim == 2 and sa.shape[0] == K // 128 and sa.shape[1] >= M
        assert sb.shape == ((N + 127) // 128, K // 128)
        D = np.zeros((M, N), np.uint16)
        cp = None
        if C is not None:
            C = _c(C, np.uint16)
            assert C.shape == (M, N)
            cp = _p(C, _u16p)
        self.lib.dg_ref_gemm_layout(_p(A, _u8p), int(a_t), _p(sa, _f32p), sa.shape[-1],
                                    _p(B, _u8p), int(b_n), _p(sb, _f32p), cp, _p(D, _u16p),
                                    M, N, K, nthreads)
        return D

    def k_grouped_tn(self, A, sa, B, sb, ks, C=None, nthreads=0):
        """K-grouped D[g] = bf16(C[g] + A_g^T B_g): A [K_all, M], B [K_all, N],
        ks the K rows of each group (multiples of 128, summing to K_all),
        sa [K_all/128, ld_sa], sb [nb, K_all/128], C bf16 bits [G, M, N] or
        None.  Returns D [G, M, N]."""
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32)
        ks = _c(ks, np.int32)
        K_all, M = A.shape
        N = B.shape[1]
        G = ks.shape[0]
        assert B.shape[0] == K_all and int(ks.sum()) == K_all
        assert np.all(ks % 128 == 0) and np.all(ks >= 0)
        assert sa.ndim == 2 and sa.shape[0] == K_all // 128 and sa.shape[1] >= M
        assert sb.shape == ((N + 127) // 128, K_all // 128)
        D = np.zeros((G, M, N), np.uint16)
        cp = None
        if C is not None:
            C = _c(C, np.uint16)
            assert C.shape == (G, M, N)
            cp = _p(C, _u16p)
        self.lib.dg_ref_k_grouped_tn(_p(A, _u8p), _p(sa, _f32p), sa.shape[-1], _p(B, _u8p),
                                     _p(sb, _f32p), cp, _p(D, _u16p), M, N, _p(ks, _i32p), G,
                                     nthreads)
        return D

    # -- UE8M0 packed scales ------------------------------------------------
    def decode_sfa(self, sfa, kb):
        """Packed UE8M0 activation scales [..., ceil(kb/4), ld] int32 ->
        fp32 [..., kb, ld]."""
        sfa = _c(sfa, np.int32)
        *lead, kbp, ld = sfa.shape
        assert kbp == (kb + 3) // 4
        flat = sfa.reshape(-1, kbp, ld)
        out = np.zeros((flat.shape[0], kb, ld), np.float32)
        for i in range(flat.shape[0]):
            src = np.ascontiguousarray(flat[i])
            dst = np.zeros((kb, ld), np.float32)
            self.lib.dg_ref_decode_sfa(_p(src, _i32p), _p(dst, _f32p), kb, ld)
            out[i] = dst
        return out.reshape(*lead, kb, ld)

    def decode_sfb(self, sfb, kb):
        """Packed UE8M0 block scales [..., nb, ceil(kb/4)] int32 -> fp32
        [..., nb, kb]."""
        sfb = _c(sfb, np.int32)
        *lead, nb, kbp = sfb.shape
        assert kbp == (kb + 3) // 4
        flat = sfb.reshape(-1, nb, kbp)
        out = np.zeros((flat.shape[0], nb, kb), np.float32)
        for i in range(flat.shape[0]):
            src = np.ascontiguousarray(flat[i])
            dst = np.zeros((nb, kb), np.float32)
            self.lib.dg_ref_decode_sfb(_p(src, _i32p), _p(dst, _f32p), nb, kb)
            out[i] = dst
        return out.reshape(*lead, nb, kb)

    def gemm_nt_ue8m0(self, A, sfa, B, sfb, nthreads=0):
        """The dense GEMM with packed UE8M0 scales: the scales decoded, then
        the same formula as gemm_nt."""
        kb = A.shape[1] // 128
        return self.gemm_nt(A, self.decode_sfa(sfa, kb), B, self.decode_sfb(sfb, kb), nthreads)

    def quantize_1x128_ue8m0(self, X, ld=None, fill=0, nthreads=0):
        """bf16 bits [G, M, K] (or [M, K]) -> (codes, packed UE8M0 scales
        [G, ceil(kb/4), ld] int32; bytes of groups past K/128 keep `fill`'s)."""
        X = _c(X, np.uint16)
        squeeze = X.ndim == 2
        if squeeze:
            X = X[None]
        G, M, K = X.shape
        ld = ld or M
        kbp = (K // 128 + 3) // 4
        Q = np.zeros((G, M, K), np.uint8)
        sfa = np.full((G, kbp, ld), fill, np.int32)
        self.lib.dg_ref_quantize_1x128_ue8m0(_p(X, _u16p), _p(Q, _u8p), _p(sfa, _i32p), G, M, K,
                                             ld, nthreads)
        return (Q[0], sfa[0]) if squeeze else (Q, sfa)

    def gemm_nt_rows(self, A, sa, B, sb, rows, nthreads=0):
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32)
        rows = _c(rows, np.int64)
        M, K = A.shape
        N = B.shape[0]
        _check_dense(A, sa, B, sb)
        assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M)
        D = np.zeros((rows.size, N), np.uint16)
        self.lib.dg_ref_gemm_nt_rows(_p(A, _u8p), _p(sa, _f32p), sa.shape[-1], _p(B, _u8p),
                                     _p(sb, _f32p), _p(D, _u16p), N, K, _p(rows, _i64p),
                                     rows.size, nthreads)
        return D

    # -- grouped ----------------------------------------------------------
    def grouped_contiguous(self, A, sa, B, sb, m_indices, rows=None, nthreads=0):
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32)
        m_indices = _c(m_indices, np.int32)
        M, K = A.shape
        G, N, K2 = B.shape
        assert K2 == K and m_indices.shape == (M,)
        assert sa.shape[0] == K // 128 and sa.shape[1] >= M
        assert sb.shape == (G, (N + 127) // 128, K // 128)
        if rows is None:
            rows_p, nrows = None, M
        else:
            rows = _c(rows, np.int64)
            assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M)
            rows_p, nrows = _p(rows, _i64p), rows.size
        D = np.zeros((nrows, N), np.uint16)
        self.lib.dg_ref_grouped_contiguous_rows(_p(A, _u8p), _p(sa, _f32p), sa.shape[-1],
                                                _p(B, _u8p), _p(sb, _f32p),
                                                _p(m_indices, _i32p), _p(D, _u16p), N, K, G,
                                                rows_p, nrows, nthreads)
        return D

    def grouped_masked(self, A, sa, B, sb, masked_m, D_init, nthreads=0):
        A = _c(A, np.uint8); B = _c(B, np.uint8)
        sa = _c(sa, np.float32); sb = _c(sb, np.float32)
        masked_m = _c(masked_m, np.int32)
        G, max_m, K = A.shape
        G2, N, K2 = B.shape
        assert G2 == G and K2 == K and masked_m.shape == (G,)
        assert sa.shape[:2] == (G, K // 128) and sa.shape[2] >= max_m
        assert sb.shape == (G, (N + 127) // 128, K // 128)
        assert masked_m.min() >= 0 and masked_m.max() <= max_m
        D = np.array(D_init, dtype=np.uint16, copy=True, order="C")
        assert D.shape == (G, max_m, N)
        self.lib.dg_ref_grouped_masked(_p(A, _u8p), _p(sa, _f32p), sa.shape[-1], _p(B, _u8p),
                                       _p(sb, _f32p), _p(masked_m, _i32p), _p(D, _u16p),
                                       G, max_m, N, K, nthreads)
        return D


    # -- activation quantiser (the step that produces A and sa) -------------
    def quantize_1x128(self, X, ld_sa=None, sa_fill=np.nan, nthreads=0):
        """X: bf16 bit patterns [M,K] or [G,M,K] (uint16).  Returns (Q, sa):
        e4m3 codes of X's shape, and fp32 scales [kb, ld_sa] ([G, kb, ld_sa]);
        scale columns m >= M keep `sa_fill`."""
        X = _c(X, np.uint16)
        squeeze = X.ndim == 2
        if squeeze:
            X = X[None]
        G, M, K = X.shape
        assert K % 128 == 0
        ld_sa = M if ld_sa is None else int(ld_sa)
        assert ld_sa >= M
        Q = np.zeros((G, M, K), np.uint8)
        sa = np.full((G, K // 128, ld_sa), sa_fill, np.float32)
        self.lib.dg_ref_quantize_1x128(_p(X, _u16p), _p(Q, _u8p), _p(sa, _f32p), G, M, K, ld_sa,
                                       nthreads)
        return (Q[0], sa[0]) if squeeze else (Q, sa)


def _check_dense(A, sa, B, sb):
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and K % 128 == 0
    assert sa.ndim == 2 and sa.shape[0] == K // 128 and sa.shape[1] >= M
    assert sb.shape == ((N + 127) // 128, K // 128)


_default = None


def default():
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def bf16_bits_to_float(bits):
    """uint16 bf16 bit patterns -> float32 values (exact)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def gemm_nt(*a, **k):
    return default().gemm_nt(*a, **k)


def gemm_nt_rows(*a, **k):
    return default().gemm_nt_rows(*a, **k)


def grouped_contiguous(*a, **k):
    return default().grouped_contiguous(*a, **k)


def grouped_masked(*a, **k):
    return default().grouped_masked(*a, **k)

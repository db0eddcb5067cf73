"""Python binding of the GB300 FP8 fine-grained-scaled GEMM library (libdg.so).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  The functions carry the C ABI's names (include/dg.h) without the
`dg_` prefix and accept either raw device addresses (int) or objects with a
`data_ptr()` method (torch tensors) for the tensor arguments, and a CUDA stream
handle (int), a torch stream, or None (torch's current stream when torch is
loaded, else the legacy default stream).

There is no fallback: if the library has not been built, `lib()` raises.
"""
import ctypes
import os

__all__ = [
    "DGError", "lib", "gemm_fp8_fp8_bf16_nt", "gemm_fp8_fp8_bf16_nt_add_c",
    "gemm_fp8_fp8_bf16_nn", "gemm_fp8_fp8_bf16_tn", "gemm_fp8_fp8_bf16_tt",
    "k_grouped_gemm_fp8_fp8_bf16_tn_contiguous", "gemm_fp8_fp8_bf16_nt_ue8m0",
    "m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0", "m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0",
    "quantize_fp8_1x128_ue8m0", "gemm_fp8_fp8_bf16_nn_ue8m0", "gemm_fp8_fp8_bf16_tn_ue8m0",
    "gemm_fp8_fp8_bf16_tt_ue8m0", "k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0",
    "m_grouped_gemm_fp8_fp8_bf16_nt_contiguous",
    "m_grouped_gemm_fp8_fp8_bf16_nt_masked", "quantize_fp8_1x128", "get_num_sms", "set_num_sms",
    "get_tma_aligned_size", "get_mk_alignment_for_contiguous_layout", "get_device_status",
    "plan_config", "num_output_tiles", "set_wait_timeout_ns", "debug_set_skip_producer",
    "debug_force_config", "debug_force_pair", "debug_force_block_scaled", "STATUS_NAMES",
    "EXPORTED_SYMBOLS",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdg.so")
#: the checked build (bounds and ring-fill checks in every kernel), loaded in
#: place of libdg.so when the environment sets DG_DEBUG=1
LIB_DEBUG_PATH = os.path.join(HERE, "libdg_debug.so")

STATUS_NAMES = {
    0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_UNSUPPORTED_SHAPE", 3: "DG_ERR_MISALIGNED",
    4: "DG_ERR_NO_DEVICE", 5: "DG_ERR_ARCH", 6: "DG_ERR_CUDA", 7: "DG_ERR_TIMEOUT",
    8: "DG_ERR_MASK_RANGE", 9: "DG_ERR_EXPERT_RANGE", 10: "DG_ERR_KS_RANGE",
    11: "DG_ERR_DEBUG_BOUNDS", 12: "DG_ERR_DEBUG_PHASE",
}

#: Every function include/dg.h declares.
EXPORTED_SYMBOLS = [
    "dg_gemm_fp8_fp8_bf16_nt", "dg_gemm_fp8_fp8_bf16_nt_add_c",
    "dg_gemm_fp8_fp8_bf16_nn", "dg_gemm_fp8_fp8_bf16_tn", "dg_gemm_fp8_fp8_bf16_tt",
    "dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous", "dg_gemm_fp8_fp8_bf16_nt_ue8m0",
    "dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0",
    "dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0", "dg_quantize_fp8_1x128_ue8m0",
    "dg_gemm_fp8_fp8_bf16_nn_ue8m0", "dg_gemm_fp8_fp8_bf16_tn_ue8m0",
    "dg_gemm_fp8_fp8_bf16_tt_ue8m0", "dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0",
    "dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous",
    "dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked", "dg_quantize_fp8_1x128", "dg_get_num_sms",
    "dg_set_num_sms",
    "dg_get_tma_aligned_size", "dg_get_mk_alignment_for_contiguous_layout",
    "dg_last_error_string", "dg_get_device_status", "dg_plan_config", "dg_plan_config_ue8m0",
    "dg_num_output_tiles",
    "dg_set_wait_timeout_ns", "dg_debug_set_skip_producer", "dg_debug_force_config",
    "dg_debug_force_pair", "dg_debug_force_block_scaled",
]


class DGError(RuntimeError):
    def __init__(self, status, detail):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.name}: {detail}")


class DGConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("block_m", "block_n", "split_k", "stages", "num_tiles", "grid", "smem_bytes",
                 "pair", "block_scaled")]


_LIB = None
_vp = ctypes.c_void_p
_i = ctypes.c_int


def lib():
    """The loaded library.  Raises if it has not been built (no fallback)."""
    global _LIB
    if _LIB is None:
        path = LIB_DEBUG_PATH if os.environ.get("DG_DEBUG", "0") not in ("", "0") else LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m moe_grouped_gemm_bf16_gb300._build`")
        L = ctypes.CDLL(path)
        L.dg_gemm_fp8_fp8_bf16_nt.argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _vp]
        L.dg_gemm_fp8_fp8_bf16_nt_add_c.argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i,
                                                    _vp]
        for name in ("nn", "tn", "tt"):
            getattr(L, "dg_gemm_fp8_fp8_bf16_" + name).argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _vp,
                                                                   _i, _i, _i, _vp]
        L.dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous.argtypes = [
            _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
        for name in ("nn", "tn", "tt"):
            getattr(L, f"dg_gemm_fp8_fp8_bf16_{name}_ue8m0").argtypes = [
                _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _vp]
        L.dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0.argtypes = [
            _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
        L.dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous.argtypes = [
            _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
        L.dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked.argtypes = [
            _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
        L.dg_quantize_fp8_1x128.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp]
        L.dg_quantize_fp8_1x128_ue8m0.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp]
        L.dg_gemm_fp8_fp8_bf16_nt_ue8m0.argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _vp]
        L.dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0.argtypes = [
            _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
        L.dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0.argtypes = [
            _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
        L.dg_get_num_sms.argtypes = []
        L.dg_set_num_sms.argtypes = [_i]
        L.dg_get_tma_aligned_size.argtypes = [_i, _i]
        L.dg_get_mk_alignment_for_contiguous_layout.argtypes = []
        L.dg_last_error_string.argtypes = []
        L.dg_last_error_string.restype = ctypes.c_char_p
        L.dg_get_device_status.argtypes = [_vp]
        L.dg_plan_config.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.POINTER(DGConfig)]
        L.dg_plan_config_ue8m0.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.POINTER(DGConfig)]
        L.dg_num_output_tiles.argtypes = [_i, _i, _i, _i]
        L.dg_num_output_tiles.restype = ctypes.c_longlong
        L.dg_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        L.dg_debug_set_skip_producer.argtypes = [_i]
        L.dg_debug_force_config.argtypes = [_i, _i]
        L.dg_debug_force_pair.argtypes = [_i]
        L.dg_debug_force_block_scaled.argtypes = [_i]
        for f in EXPORTED_SYMBOLS:
            if f not in ("dg_last_error_string", "dg_num_output_tiles"):
                getattr(L, f).restype = _i
        _LIB = L
    return _LIB


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s):
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream)
        except Exception:  # pragma: no cover
            pass
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(status):
    if status != 0:
        raise DGError(status, lib().dg_last_error_string().decode())


def gemm_fp8_fp8_bf16_nt(A, sa, ld_sa, B, sb, D, M, N, K, stream=None):
    """D[M,N] = bf16(sum_g (A_g B_g^T) sa sb); see dg_gemm_fp8_fp8_bf16_nt."""
    _check(lib().dg_gemm_fp8_fp8_bf16_nt(_ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb), _ptr(D),
                                         M, N, K, _stream(stream)))


def gemm_fp8_fp8_bf16_nt_add_c(A, sa, ld_sa, B, sb, C, D, M, N, K, stream=None):
    """D[M,N] = bf16(C + sum_g (A_g B_g^T) sa sb); C may be D."""
    _check(lib().dg_gemm_fp8_fp8_bf16_nt_add_c(_ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb),
                                               _ptr(C), _ptr(D), M, N, K, _stream(stream)))


def gemm_fp8_fp8_bf16_nn(A, sa, ld_sa, B, sb, D, M, N, K, C=None, stream=None):
    """D[M,N] = bf16(C + A @ B): A [M,K], B [K,N]; C optional (may be D)."""
    _check(lib().dg_gemm_fp8_fp8_bf16_nn(_ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb), _ptr(C),
                                         _ptr(D), M, N, K, _stream(stream)))


def gemm_fp8_fp8_bf16_tn(A, sa, ld_sa, B, sb, D, M, N, K, C=None, stream=None):
    """D[M,N] = bf16(C + A^T @ B): A [K,M], B [K,N]; C optional (may be D)."""
    _check(lib().dg_gemm_fp8_fp8_bf16_tn(_ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb), _ptr(C),
                                         _ptr(D), M, N, K, _stream(stream)))


def gemm_fp8_fp8_bf16_tt(A, sa, ld_sa, B, sb, D, M, N, K, C=None, stream=None):
    """D[M,N] = bf16(C + A^T @ B^T): A [K,M], B [N,K]; C optional (may be D)."""
    _check(lib().dg_gemm_fp8_fp8_bf16_tt(_ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb), _ptr(C),
                                         _ptr(D), M, N, K, _stream(stream)))


def k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(A, sa, ld_sa, B, sb, D, ks, num_groups, M, N,
                                              K_total, C=None, stream=None):
    """D[g] = bf16(C[g] + A_g^T B_g) over each group's K rows: A [K_total,M],
    B [K_total,N], ks int32 [G] on the device, D (and C) [G,M,N]."""
    _check(lib().dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(
        _ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb), _ptr(C), _ptr(D), _ptr(ks), num_groups, M, N,
        K_total, _stream(stream)))


def m_grouped_gemm_fp8_fp8_bf16_nt_contiguous(A, sa, ld_sa, B, sb, D, m_indices, M_total, N, K,
                                              num_groups, stream=None):
    _check(lib().dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous(
        _ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb), _ptr(D), _ptr(m_indices), M_total, N, K,
        num_groups, _stream(stream)))


def m_grouped_gemm_fp8_fp8_bf16_nt_masked(A, sa, ld_sa, B, sb, D, masked_m, num_groups, max_m,
                                          N, K, expected_m, stream=None):
    _check(lib().dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked(
        _ptr(A), _ptr(sa), ld_sa, _ptr(B), _ptr(sb), _ptr(D), _ptr(masked_m), num_groups, max_m,
        N, K, expected_m, _stream(stream)))


def gemm_fp8_fp8_bf16_nt_ue8m0(A, sfa, ld_sfa, B, sfb, D, M, N, K, stream=None):
    """The dense GEMM with packed UE8M0 scales (int32 sfa [ceil(K/512), ld_sfa],
    sfb [ceil(N/128), ceil(K/512)])."""
    _check(lib().dg_gemm_fp8_fp8_bf16_nt_ue8m0(_ptr(A), _ptr(sfa), ld_sfa, _ptr(B), _ptr(sfb),
                                               _ptr(D), M, N, K, _stream(stream)))


def m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(A, sfa, ld_sfa, B, sfb, D, m_indices, M_total,
                                                    N, K, num_groups, stream=None):
    _check(lib().dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(
        _ptr(A), _ptr(sfa), ld_sfa, _ptr(B), _ptr(sfb), _ptr(D), _ptr(m_indices), M_total, N, K,
        num_groups, _stream(stream)))


def m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(A, sfa, ld_sfa, B, sfb, D, masked_m, num_groups,
                                                max_m, N, K, expected_m, stream=None):
    _check(lib().dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(
        _ptr(A), _ptr(sfa), ld_sfa, _ptr(B), _ptr(sfb), _ptr(D), _ptr(masked_m), num_groups,
        max_m, N, K, expected_m, _stream(stream)))


def _layout_ue8m0(name):
    def fn(A, sfa, ld_sfa, B, sfb, D, M, N, K, C=None, stream=None):
        _check(getattr(lib(), f"dg_gemm_fp8_fp8_bf16_{name}_ue8m0")(
            _ptr(A), _ptr(sfa), ld_sfa, _ptr(B), _ptr(sfb), _ptr(C), _ptr(D), M, N, K,
            _stream(stream)))
    fn.__name__ = f"gemm_fp8_fp8_bf16_{name}_ue8m0"
    fn.__doc__ = f"The {name} dense GEMM with packed UE8M0 scales; C optional (may be D)."
    return fn


gemm_fp8_fp8_bf16_nn_ue8m0 = _layout_ue8m0("nn")
gemm_fp8_fp8_bf16_tn_ue8m0 = _layout_ue8m0("tn")
gemm_fp8_fp8_bf16_tt_ue8m0 = _layout_ue8m0("tt")


def k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0(A, sfa, ld_sfa, B, sfb, D, ks, num_groups, M,
                                                    N, K_total, C=None, stream=None):
    """The K-grouped tn GEMM with packed UE8M0 scales (sfa [K_total/512, ld_sfa],
    sfb [ceil(N/128), K_total/512], int32)."""
    _check(lib().dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0(
        _ptr(A), _ptr(sfa), ld_sfa, _ptr(B), _ptr(sfb), _ptr(C), _ptr(D), _ptr(ks), num_groups, M,
        N, K_total, _stream(stream)))


def quantize_fp8_1x128_ue8m0(X, Q, sfa, num_groups, M, K, ld_sfa, stream=None):
    """bf16 X [G,M,K] -> e4m3 Q and packed UE8M0 scales sfa int32 [G, ceil(K/512), ld_sfa]."""
    _check(lib().dg_quantize_fp8_1x128_ue8m0(_ptr(X), _ptr(Q), _ptr(sfa), num_groups, M, K,
                                             ld_sfa, _stream(stream)))


def quantize_fp8_1x128(X, Q, sa, num_groups, M, K, ld_sa, stream=None):
    """Per-token 1x128 FP8 quantisation of bf16 X [G,M,K] into e4m3 Q and fp32
    sa [G,K/128,ld_sa]; see dg_quantize_fp8_1x128."""
    _check(lib().dg_quantize_fp8_1x128(_ptr(X), _ptr(Q), _ptr(sa), num_groups, M, K, ld_sa,
                                       _stream(stream)))


def get_num_sms():
    return int(lib().dg_get_num_sms())


def set_num_sms(n):
    _check(lib().dg_set_num_sms(int(n)))


def get_tma_aligned_size(mn, elem_bytes):
    return int(lib().dg_get_tma_aligned_size(int(mn), int(elem_bytes)))


def get_mk_alignment_for_contiguous_layout():
    return int(lib().dg_get_mk_alignment_for_contiguous_layout())


def get_device_status(stream=None):
    """Status code (int) of the device status word, which is then cleared."""
    return int(lib().dg_get_device_status(_stream(stream)))


def plan_config(kind, m, n, k, num_groups=1, num_sms=152, ue8m0=False):
    cfg = DGConfig()
    fn = lib().dg_plan_config_ue8m0 if ue8m0 else lib().dg_plan_config
    _check(fn(int(kind), int(m), int(n), int(k), int(num_groups), int(num_sms), ctypes.byref(cfg)))
    return {f: getattr(cfg, f) for f, _ in DGConfig._fields_}


def num_output_tiles(m, n, block_m, block_n):
    return int(lib().dg_num_output_tiles(int(m), int(n), int(block_m), int(block_n)))


def set_wait_timeout_ns(ns):
    _check(lib().dg_set_wait_timeout_ns(int(ns)))


def debug_set_skip_producer(on):
    _check(lib().dg_debug_set_skip_producer(1 if on else 0))


def debug_force_config(block_n=0, split_k=0):
    _check(lib().dg_debug_force_config(int(block_n), int(split_k)))


def debug_force_pair(mode=-1):
    _check(lib().dg_debug_force_pair(int(mode)))


def debug_force_block_scaled(mode=-1):
    """-1 heuristic, 0 never, 1 only the block-scaled kernels (packed UE8M0 forms)."""
    _check(lib().dg_debug_force_block_scaled(int(mode)))

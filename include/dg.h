/*
 * dg.h - C ABI of the GB300 (sm_103a) FP8 fine-grained-scaled GEMM library.
 *
 * Every GEMM entry point computes, for the rows it covers,
 *
 *   D[m,n] = bf16( [C[m,n] +] sum over K groups g of (A_g . B_g^T)[m,n] * sa[m,g] * sb[n/128,g] )
 *
 * with A e4m3 (OCP "E4M3FN" codes, one byte each), B e4m3, both row-major with
 * K innermost ("NT": LHS not transposed, RHS transposed) unless the entry point
 * names another layout, g a 128-wide slice of K, one scale per row per K group
 * for A and one per 128x128 block for B (fp32, or packed UE8M0 in the "_ue8m0"
 * entry points), an optional bf16 addend C where the entry point takes one, and
 * a bf16 (round-to-nearest-even) output.  This is the GEMM of DeepGEMM
 * (es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de layout";
 * the original names follow the release as listed on deepep.org/zh/deepgemm,
 * "接口设计").  The layouts below are those of the NT entry points; the others
 * state theirs where they are declared.
 *
 * Conventions shared by all entry points
 *  - All tensor arguments are DEVICE pointers owned by the caller; the library
 *    keeps no reference after the call returns and allocates nothing.
 *  - A, B, D and sa must be 16-byte aligned; sb 4-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  A call never synchronises, never reads device memory
 *    from the host and never allocates, so it can be captured in a CUDA graph.
 *  - Argument errors are reported by the return value before anything is
 *    launched; dg_last_error_string() gives the detail.  Errors found on the
 *    device (a masked_m out of range, a contiguous block that mixes experts, a
 *    bad K-grouped ks entry, an internal wait that timed out) are recorded in a
 *    device status word read by dg_get_device_status().  There is one such
 *    word per device, shared by every stream and every call on that device.
 *  - Bounded waits: every wait inside a kernel (for an operand tile, a tensor-
 *    memory accumulator, a peer CTA) gives up after a time limit, 2 s unless
 *    dg_set_wait_timeout_ns() sets another.  A kernel whose wait gives up
 *    records DG_ERR_TIMEOUT in the status word and finishes WITHOUT its
 *    result (D is left partly written); the GEMM call itself has already
 *    returned DG_OK.  A call that can legitimately take longer than the limit
 *    (a very large problem on a GPU time-sliced with other work) needs a
 *    larger limit, and callers that must know whether a result is complete
 *    poll dg_get_device_status().
 *  - The current CUDA device must be a compute capability 10.3 GPU (GB300).
 *  - Checked build: the same ABI is also built as libdg_debug.so (every
 *    kernel compiled with DG_DEBUG=1).  Before each TMA load and each plain
 *    global store its kernels check the coordinates against the tensors'
 *    extents, and after each wait on a producer -> consumer ring they check
 *    that the slot holds the fill they expect.  A failed check skips the
 *    access, aborts the kernel through the bounded-wait path and records
 *    DG_ERR_DEBUG_BOUNDS or DG_ERR_DEBUG_PHASE in the status word; nothing
 *    traps.  It is slower and meant for tests.
 *
 * Layouts
 *  - A  : [M][K] bytes (masked form: [G][max_m][K]).
 *  - sa : fp32, K-group-major ("transposed", TMA-aligned):
 *         sa[g * ld_sa + m], g < K/128, ld_sa >= M (masked: max_m), ld_sa % 4 == 0.
 *         Masked form: sa[(grp * K/128 + g) * ld_sa + m].
 *  - B  : [N][K] bytes (grouped forms: [G][N][K]).
 *  - sb : fp32 [ceil(N/128)][K/128] (grouped forms: [G][ceil(N/128)][K/128]);
 *         sb[(n/128) * (K/128) + g].
 *  - D  : bf16 bit patterns [M][N] (masked form: [G][max_m][N]).
 *  - Shape limits: K % 128 == 0, 128 <= K <= 65536; N % 16 == 0; N >= 16.
 */
#ifndef DG_H_
#define DG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dg_status {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad group count */
  DG_ERR_UNSUPPORTED_SHAPE = 2, /* K or N outside the shape limits above */
  DG_ERR_MISALIGNED = 3,        /* pointer or ld_sa alignment */
  DG_ERR_NO_DEVICE = 4,         /* no CUDA device available */
  DG_ERR_ARCH = 5,              /* current device is not compute capability 10.3 */
  DG_ERR_CUDA = 6,              /* a CUDA runtime/driver call failed */
  DG_ERR_TIMEOUT = 7,           /* device: an internal wait gave up */
  DG_ERR_MASK_RANGE = 8,        /* device: masked_m[g] outside [0, max_m] (clamped) */
  DG_ERR_EXPERT_RANGE = 9,      /* device: m_indices outside [-1, G) or a 128-row block mixes experts */
  DG_ERR_KS_RANGE = 10,         /* device: ks[g] negative, not a multiple of 128, or past K_total */
  DG_ERR_DEBUG_BOUNDS = 11,     /* device, checked build only: an access outside a tensor (skipped) */
  DG_ERR_DEBUG_PHASE = 12       /* device, checked build only: a ring slot held another fill */
} dg_status;

/* Dense GEMM (DeepGEMM "gemm_fp8_fp8_bf16_nt", deepep.org/zh/deepgemm, "接口设计").
 * A [M][K], sa [K/128][ld_sa], B [N][K], sb [ceil(N/128)][K/128], D [M][N].
 * M == 0 is a no-op. */
dg_status dg_gemm_fp8_fp8_bf16_nt(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, void* D, int M, int N, int K, void* stream);

/* The same dense GEMM with an addend: D = C + A @ B^T (the naming convention
 * D = C + A @ B of es.news.hada.io/topic?id=19459, "Interfaz GEMM y
 * restricciones de layout").  C is bf16 [M][N] row-major, 16-byte aligned,
 * caller-owned; it may be D itself (each element is read before it is
 * written, by the same thread).  Per element, the C value is added in fp32 to
 * the fp32 sum of the scaled K groups, and the total is rounded once to bf16.
 * Everything else, errors included, is as for dg_gemm_fp8_fp8_bf16_nt; a null
 * C is DG_ERR_INVALID_ARG. */
dg_status dg_gemm_fp8_fp8_bf16_nt_add_c(const void* A, const float* sa, int ld_sa, const void* B,
                                        const float* sb, const void* C, void* D, int M, int N,
                                        int K, void* stream);

/* The dense GEMM in the other storage layouts (DeepGEMM's fp8_gemm_{nn, tn, tt},
 * es.news.hada.io/topic?id=19459, "Dense y Grouped GEMM"; all four layouts
 * on SM100, "Interfaz GEMM y restricciones de layout").  The letters say
 * whether each stored operand enters D = C + A @ B transposed:
 *   nn  A [M][K], B [K][N]      tn  A [K][M], B [K][N]      tt  A [K][M], B [N][K]
 * (nt, above: A [M][K], B [N][K]).  The scales do not move with the operands:
 * sa [K/128][ld_sa] one per (row m, K group), sb [ceil(N/128)][K/128] one per
 * 128 x 128 block of (n, k); D and the optional addend C (null: none; may be
 * D itself) bf16 [M][N].  Per element the result is
 *   D[m,n] = bf16( C[m,n] + sum_g (sum_{k in g} A(m,k) B(n,k)) sa[g][m] sb[n/128][g] ).
 * Requirements as for dg_gemm_fp8_fp8_bf16_nt, and M a multiple of 16 when A
 * is stored [K][M] (a row of it is M bytes), else DG_ERR_UNSUPPORTED_SHAPE. */
dg_status dg_gemm_fp8_fp8_bf16_nn(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, const void* C, void* D, int M, int N, int K,
                                  void* stream);
dg_status dg_gemm_fp8_fp8_bf16_tn(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, const void* C, void* D, int M, int N, int K,
                                  void* stream);
dg_status dg_gemm_fp8_fp8_bf16_tt(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, const void* C, void* D, int M, int N, int K,
                                  void* stream);

/* K-grouped GEMM for the MoE weight gradient (DeepGEMM
 * "k_grouped_fp8_gemm_tn_contiguous", es.news.hada.io/topic?id=19459, "Dense
 * y Grouped GEMM": M and N fixed, the groups concatenated along K).  Group g
 * owns the K rows [k0_g, k0_g + ks[g]), k0_g = ks[0] + ... + ks[g-1]:
 *   D[g][m][n] = bf16( C[g][m][n] + sum over the K groups j of group g of
 *                      (sum_{k in j} A[k][m] B[k][n]) sa[j][m] sb[n/128][j] )
 *   A   e4m3 [K_total][M] ("t"), B e4m3 [K_total][N] ("n")
 *   sa  fp32 [K_total/128][ld_sa], sb fp32 [ceil(N/128)][K_total/128]
 *   C   bf16 [num_groups][M][N] or null (none); it may be D itself
 *   D   bf16 [num_groups][M][N]
 *   ks  int32 [num_groups] on the device (read by the kernel, never by the
 *       host, so a captured graph follows new values): each a multiple of 128,
 *       >= 0, summing to at most K_total.  A group with ks[g] = 0 gets D = C
 *       (or +0).  A bad entry is clamped (to whole K groups within K_total)
 *       and reported as DG_ERR_KS_RANGE by dg_get_device_status.
 * Requirements (host-checked): 1 <= num_groups <= 1024; K_total a positive
 * multiple of 128 up to 65536; M and N multiples of 16; ld_sa >= M, a
 * multiple of 4; A, B, C, D, sa 16-byte aligned, sb and ks 4-byte aligned.
 * M == 0 is a no-op. */
dg_status dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(const void* A, const float* sa, int ld_sa,
                                                       const void* B, const float* sb,
                                                       const void* C, void* D, const int32_t* ks,
                                                       int num_groups, int M, int N, int K_total,
                                                       void* stream);

/* M-grouped GEMM, contiguous layout (DeepGEMM "m_grouped_gemm_fp8_fp8_bf16_nt_contiguous";
 * es.news.hada.io/topic?id=19459, "Dense y Grouped GEMM": the experts' rows are
 * concatenated along M, each expert's segment aligned to the M block size).
 * A [M_total][K], sa [K/128][ld_sa], B [num_groups][N][K], sb [num_groups][ceil(N/128)][K/128],
 * D [M_total][N], m_indices int32 [M_total] on the device: the expert of each row,
 * or -1 for a padding row.  Padding rows of D are written as +0.
 * M_total % 128 == 0 (dg_get_mk_alignment_for_contiguous_layout()); every 128-row
 * block holds rows of one expert, optionally followed by padding rows; a block
 * whose first row is -1 is all padding. */
dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous(const void* A, const float* sa, int ld_sa,
                                                       const void* B, const float* sb, void* D,
                                                       const int32_t* m_indices, int M_total,
                                                       int N, int K, int num_groups,
                                                       void* stream);

/* M-grouped GEMM, masked layout (DeepGEMM "m_grouped_gemm_fp8_fp8_bf16_nt_masked";
 * es.news.hada.io/topic?id=19459, "Dense y Grouped GEMM": for decoding under CUDA
 * graphs, where the host does not know how many tokens each expert got).
 * A [G][max_m][K], sa [G][K/128][ld_sa], B [G][N][K], sb [G][ceil(N/128)][K/128],
 * D [G][max_m][N], masked_m int32 [G] on the device: rows m < masked_m[g] of group g
 * are computed; the other rows of D are not written.  The host never reads
 * masked_m.  expected_m is a hint for the tile-size choice only; results never
 * depend on it.  1 <= num_groups <= 1024. */
dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked(const void* A, const float* sa, int ld_sa,
                                                   const void* B, const float* sb, void* D,
                                                   const int32_t* masked_m, int num_groups,
                                                   int max_m, int N, int K, int expected_m,
                                                   void* stream);

/* The same GEMMs with packed UE8M0 scales, the scale format of DeepGEMM's SM100
 * kernels (es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de
 * layout": packed UE8M0, four per 32-bit integer).  A UE8M0 code e is the
 * scale 2^(e - 127) (0xFF: NaN); the four K groups 4i .. 4i+3 share one
 * int32 word, group 4i + j in bits 8j .. 8j+7.
 *   sfa  int32 [ceil(K/512)][ld_sfa] (masked: [G][ceil(K/512)][ld_sfa]): word
 *        (i, m) holds row m's scales of K groups 4i ..; ld_sfa >= rows, a
 *        multiple of 4; 16-byte aligned
 *   sfb  int32 [ceil(N/128)][ceil(K/512)] (grouped: [G][ceil(N/128)][ceil(K/512)]):
 *        word (b, i) holds the 128-row block b's scales of K groups 4i ..
 * Every other argument, the result's formula and the errors are those of the
 * fp32-scale entry point of the same name without "_ue8m0"; the scales are
 * decoded exactly (every UE8M0 value but NaN is an fp32 value).  Bytes of K
 * groups >= K/128 in the last word are never read. */
dg_status dg_gemm_fp8_fp8_bf16_nt_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, void* D, int M, int N,
                                        int K, void* stream);
/* nn / tn / tt and K-grouped with packed UE8M0 scales: the scales are packed
 * as above (sfa [ceil(K/512)][ld_sfa] per row m, sfb [ceil(N/128)][ceil(K/512)]
 * per 128-row block of B's n; K-grouped: K = K_total), everything else as in
 * the fp32-scale entry point of the same name. */
dg_status dg_gemm_fp8_fp8_bf16_nn_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, const void* C, void* D,
                                        int M, int N, int K, void* stream);
dg_status dg_gemm_fp8_fp8_bf16_tn_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, const void* C, void* D,
                                        int M, int N, int K, void* stream);
dg_status dg_gemm_fp8_fp8_bf16_tt_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, const void* C, void* D,
                                        int M, int N, int K, void* stream);
dg_status dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0(
    const void* A, const int32_t* sfa, int ld_sfa, const void* B, const int32_t* sfb,
    const void* C, void* D, const int32_t* ks, int num_groups, int M, int N, int K_total,
    void* stream);
dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(
    const void* A, const int32_t* sfa, int ld_sfa, const void* B, const int32_t* sfb, void* D,
    const int32_t* m_indices, int M_total, int N, int K, int num_groups, void* stream);
dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(
    const void* A, const int32_t* sfa, int ld_sfa, const void* B, const int32_t* sfb, void* D,
    const int32_t* masked_m, int num_groups, int max_m, int N, int K, int expected_m,
    void* stream);

/* Per-token 1x128 FP8 quantisation of a bf16 activation matrix: the step that
 * produces the left operand A and its scales sa in the layout the GEMMs above
 * read (es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de
 * layout": LHS scales fp32, transposed and TMA-aligned; the pages leave the
 * conversion itself to the caller, so its arithmetic is this library's
 * reading).  For each row m and 128-wide K group g, in fp32:
 *   a = max(max_k |X[m,k]|, 1e-4);  sa[g][m] = a / 448;
 *   Q[m,k] = e4m3(X[m,k] * (448 / a)), rounded to nearest even, saturating
 *   at +-448 (so the group's largest |X| becomes code magnitude 448).
 *   X   bf16 [num_groups][M][K] row-major (num_groups = 1 for a dense matrix,
 *       or G for the masked layout [G][max_m][K] with M = max_m); finite values
 *   Q   e4m3 codes, same shape as X
 *   sa  fp32 [num_groups][K/128][ld_sa]; columns m < M are written, the
 *       others (ld_sa - M of them per row) are left as they were
 * Requirements (checked on the host; on failure nothing is launched):
 * non-null pointers, num_groups >= 1, M >= 0, ld_sa >= M (else
 * DG_ERR_INVALID_ARG); K a positive multiple of 128, num_groups * M * K/128
 * < 2^31, K/128 <= 65535 and num_groups <= 65535 (else
 * DG_ERR_UNSUPPORTED_SHAPE); ld_sa a multiple of 4 and X, Q, sa
 * 16-byte aligned (else DG_ERR_MISALIGNED).  M = 0 does nothing.
 * Asynchronous on `stream`; device memory is caller-owned; no allocation, no
 * host synchronisation. */
dg_status dg_quantize_fp8_1x128(const void* X, void* Q, float* sa, int num_groups, int M, int K,
                                int ld_sa, void* stream);

/* The quantiser with UE8M0 scales for the "_ue8m0" GEMMs: per row m and K
 * group g, in fp32, a = max(max_k |X[m,k]|, 1e-4); t = a / 448; s = the
 * smallest power of two >= t; Q[m,k] = e4m3(X[m,k] / s) (round to nearest
 * even, saturating; the division by s is exact); the code 127 + log2(s) is
 * written to byte g % 4 of word sfa[z][g / 4][m] (int32 [num_groups][ceil(K/512)]
 * [ld_sfa]).  Bytes of K groups >= K/128 and columns m >= M are left as they
 * were.  Requirements and errors as for dg_quantize_fp8_1x128 (ld_sfa in place
 * of ld_sa). */
dg_status dg_quantize_fp8_1x128_ue8m0(const void* X, void* Q, int32_t* sfa, int num_groups,
                                      int M, int K, int ld_sfa, void* stream);

/* Maximum number of SMs the kernels may use (DeepGEMM set_num_sms / get_num_sms,
 * es.news.hada.io/topic?id=19459, "Utilidades y variables de entorno").
 * dg_set_num_sms(0) restores "all SMs of the device"; a value above the device's
 * SM count is rejected with DG_ERR_INVALID_ARG when a device is present.
 * dg_get_num_sms() returns the limit in force (the device's SM count by default,
 * 0 when no device is present and no limit was set). */
int dg_get_num_sms(void);
dg_status dg_set_num_sms(int num_sms);

/* Smallest count >= mn whose size in bytes (count * elem_bytes) is a multiple of
 * 16: the TMA-aligned leading dimension of the transposed scales (DeepGEMM
 * get_tma_aligned_size, same section).  Returns -1 for mn < 0 or elem_bytes <= 0. */
int dg_get_tma_aligned_size(int mn, int elem_bytes);

/* Row alignment of each expert's segment in the contiguous layout: the M block
 * size, 128 (DeepGEMM get_mk_alignment_for_contiguous_layout, same section). */
int dg_get_mk_alignment_for_contiguous_layout(void);

/* Human-readable detail of the last error returned on this thread ("" if none). */
const char* dg_last_error_string(void);

/* Waits for `stream`, then returns and clears the device status word of the
 * current device: DG_OK, or the first device-side error recorded since the last
 * call (DG_ERR_TIMEOUT, DG_ERR_MASK_RANGE, DG_ERR_EXPERT_RANGE, DG_ERR_KS_RANGE).
 * The word is per device and shared across streams: an error raised by a
 * kernel on any stream of the device is reported here, and work still running
 * on other streams may raise one after this call returns.  The read and the
 * clear are one atomic exchange on the device (a one-thread kernel on
 * `stream`), so no error is lost between them. */
dg_status dg_get_device_status(void* stream);

/* Tile configuration the library would choose (heuristic; no device needed).
 * kind: 0 dense (nt), 1 contiguous, 2 masked, 3 K-grouped (tn).  m is M
 * (dense, K-grouped), M_total (contiguous) or expected_m (masked); k is K
 * (K-grouped: K_total, planned as num_groups equal groups).  num_sms is the
 * SM count to plan for.
 * With a GB300 as the current device (and num_sms at most its SM count), the
 * clusters that fit at once are the device's, so the result is the
 * configuration a launch on num_sms SMs takes; without one, num_sms / S
 * clusters of S CTAs are assumed to fit. */
typedef struct dg_config {
  int block_m;      /* output tile height: 128, or 256 in the CTA-pair form */
  int block_n;      /* output tile width */
  int split_k;      /* CTAs per cluster sharing one tile's K groups (dense only) */
  int stages;       /* depth of the shared-memory ring */
  int num_tiles;    /* output tiles (masked: from expected_m) */
  int grid;         /* CTAs launched */
  int smem_bytes;   /* dynamic shared memory per CTA */
  int pair;         /* 1: CTA-pair form (a 2-CTA cluster computes each block_m = 256 tile) */
  int block_scaled; /* 1: the block-scaled kernel (packed UE8M0 scales applied by the MMA) */
} dg_config;
dg_status dg_plan_config(int kind, int m, int n, int k, int num_groups, int num_sms,
                         dg_config* out);

/* The same for the "_ue8m0" entry points of each kind (packed UE8M0 scales),
 * which choose between the block-scaled kernels and the promotion kernels'
 * packed-scale twins (block_scaled says which). */
dg_status dg_plan_config_ue8m0(int kind, int m, int n, int k, int num_groups, int num_sms,
                               dg_config* out);

/* Number of BLOCK_M x BLOCK_N output tiles of an M x N output (the unit of the
 * persistent scheduler; deepep.org/zh/deepgemm, "核心优化技术", unaligned block
 * sizes). Returns -1 for non-positive block sizes. */
long long dg_num_output_tiles(int m, int n, int block_m, int block_n);

/* Upper bound, in nanoseconds, of every internal wait of the kernels; past it a
 * kernel records DG_ERR_TIMEOUT and finishes without its result.  0 restores the
 * default (2 s). */
dg_status dg_set_wait_timeout_ns(unsigned long long ns);

/* Test hook for the failure path: when nonzero, the next launches run with the
 * TMA producer switched off, so that their waits run out (DG_ERR_TIMEOUT).  Use
 * only together with a short dg_set_wait_timeout_ns(). */
dg_status dg_debug_set_skip_producer(int on);

/* Test and benchmark hook: force the tile width (block_n) and the K split
 * (split_k, 1..8) of the following launches; 0 leaves that choice to the
 * heuristic.  A forced configuration the shape cannot use makes the GEMM calls
 * return DG_ERR_UNSUPPORTED_SHAPE.  The environment variable
 * DG_FORCE_CONFIG="block_n,split_k" sets the same at start-up. */
dg_status dg_debug_force_config(int block_n, int split_k);

/* Test and benchmark hook: -1 (default) lets the heuristic decide whether a
 * dense GEMM runs in the CTA-pair form (256-row tiles computed by a 2-CTA
 * cluster with one shared MMA), and likewise the masked form (256-row blocks
 * of a group); 0 never, 1 always (the contiguous form and the MN-major layouts
 * have no pair kernel, so 1 makes them return DG_ERR_UNSUPPORTED_SHAPE).  The
 * environment variable DG_FORCE_PAIR=0|1 sets the same before the first call. */
dg_status dg_debug_force_pair(int mode);

/* Test and benchmark hook for the packed-UE8M0 entry points: -1 (default)
 * lets the heuristic choose between the block-scaled kernels (the tensor
 * cores apply the UE8M0 scales, tcgen05.mma kind::mxf8f6f4 with block
 * scaling, and accumulate all of a tile's K in tensor memory) and the
 * kernels that decode the scales into the per-K-group promotion (which also
 * hold the K-split forms); 0 never the block-scaled ones, 1 only those (a
 * shape or forced configuration without one returns DG_ERR_UNSUPPORTED_SHAPE).
 * Results agree within the stated tolerance either way.  The environment
 * variable DG_FORCE_BLOCK_SCALED=0|1 sets the same before the first call. */
dg_status dg_debug_force_block_scaled(int mode);

#ifdef __cplusplus
}
#endif

#endif /* DG_H_ */

// Launch parameters shared by the host launcher and the kernels.
#pragma once
#include <cstdint>

namespace dgk {

// Which form of the GEMM a launch computes (DeepGEMM, es.news.hada.io/topic?id=19459,
// "Dense y Grouped GEMM"): dense, M-grouped contiguous, M-grouped masked, and
// the K-grouped form of the MoE weight gradient (groups concatenated along K).
enum Mode : int { kDense = 0, kContiguous = 1, kMasked = 2, kKGrouped = 3 };

// Operand storage (same page, "Interfaz GEMM y restricciones de layout": the
// nt / nn / tn / tt layouts).  Bit 0: A stored [K][M] ("t"), else [M][K];
// bit 1: B stored [K][N] ("n"), else [N][K].  A [K][M] operand is MN-major
// in shared memory, which tcgen05 reads for 8-bit types as well.
enum Layout : int { kNT = 0, kTT = 1, kNN = 2, kTN = 3 };

constexpr int BLOCK_M = 128;  // rows of A per tile (one tcgen05 M=128 MMA)
constexpr int BLOCK_K = 128;  // one K group: the granularity of both scale factors
// Promotion warpgroups (each covers all 128 tile rows and 1/PROMO_WG of the
// columns).  Warpgroup 0: warp 0 TMA, warps 1.. MMA issue.
#ifndef DG_PROMO_WG
#define DG_PROMO_WG 2
#endif
constexpr int PROMO_WG = DG_PROMO_WG;
static_assert(PROMO_WG == 2 || PROMO_WG == 4, "two or four promotion warpgroups");
constexpr int NUM_THREADS = 128 * (1 + PROMO_WG);
constexpr int NUM_PROMO_WARPS = 4 * PROMO_WG;
// 32-column TMEM chunks a promotion warp loads per tcgen05.wait::ld
#ifndef DG_PROMO_LB
#define DG_PROMO_LB 2
#endif
constexpr int PROMO_LB = DG_PROMO_LB;
// MMA issuer warps (warps 1..NUM_ISSUERS of warpgroup 0), taking K groups in turn
#ifndef DG_NUM_ISSUERS
#define DG_NUM_ISSUERS 2
#endif
constexpr int NUM_ISSUERS = DG_NUM_ISSUERS;
static_assert(NUM_ISSUERS == 1 || NUM_ISSUERS == 2, "the issuer count must divide every NBUF");
// Activation-scale ring: each slot holds the scales of SA_GROUPS consecutive K
// groups (one TMA load, one full/empty barrier round trip per slot)
constexpr int SA_GROUPS = 4;
constexpr int SA_SLOTS = 4;
constexpr int MAX_GROUPS_MASKED = 1024;
constexpr int MAX_GROUPS_KGROUPED = 1024;
constexpr int MAX_KB = 512;   // K <= 65536
constexpr int MAX_SPLIT = 8;  // CTAs per cluster in the K-split form
// 32-bit words of one of a CTA's two B-scale buffers: a tile's [3][K/128]
// scales (per K group), or the 16-byte aligned span of global memory holding
// the rows of its (up to 3) 128-column blocks (fp32: K/128 words per row,
// packed UE8M0: K/512), which starts up to 3 words before the first row and
// ends up to 3 words after the last.
__host__ __device__ constexpr int sb_buf_words(int kb) { return (3 * kb + 8 + 3) & ~3; }

// Checked build (compiled with -DDG_DEBUG=1; the library libdg_debug.so):
// before every TMA load and every plain global store the kernels check the
// coordinates against the tensors' extents, and after every wait on a
// producer -> consumer ring barrier the consumer checks that the slot holds
// the fill it expects (a wait that passed a phase early would see another).
// A failed check records ST_DEBUG_BOUNDS / ST_DEBUG_PHASE in the status word,
// skips the access and aborts the CTA (the bounded-wait path); nothing traps.
#ifndef DG_DEBUG
#define DG_DEBUG 0
#endif
constexpr bool kDebug = DG_DEBUG != 0;

// Device status word values (first error wins).
constexpr unsigned int ST_OK = 0;
constexpr unsigned int ST_TIMEOUT = 7;      // an mbarrier wait gave up
constexpr unsigned int ST_MASK_RANGE = 8;   // masked_m[g] outside [0, max_m]; clamped
constexpr unsigned int ST_EXPERT_RANGE = 9; // m_indices out of range or a block mixes experts
constexpr unsigned int ST_KS_RANGE = 10;    // ks[g] negative, not a multiple of 128, or past K
constexpr unsigned int ST_DEBUG_BOUNDS = 11; // checked build: an access outside a tensor, skipped
constexpr unsigned int ST_DEBUG_PHASE = 12;  // checked build: a ring slot held another fill

// Debug flags (tests of the failure path only).
constexpr unsigned int DBG_SKIP_PRODUCER = 1u;  // the TMA warp issues nothing

struct Params {
  int M;           // dense: rows of A/D; contiguous: M_total; masked: max_m
  int N;
  int K;
  int kb;          // K / 128
  int nb;          // ceil(N / 128): B scale blocks per group
  int num_groups;  // experts (grouped) or 1
  int num_m_blocks;  // dense: ceil(M/128); contiguous: M_total/128; masked: computed on device
  int num_n_blocks;  // ceil(N / BLOCK_N)
  int raster_m;      // M blocks per raster band
  int split_k;       // CTAs per cluster, each taking a slice of the K groups
  const float* sb;             // [G][nb][kb] fp32, or [G][nb][kbp] packed UE8M0 words (the
                               // instance's SFP parameter says which)
  int kbp;                     // ceil(kb / 4): packed words per row of scales
  const void* sa_packed;       // packed UE8M0 activation scales [z][kbp][ld_sa] (block-scaled
                               // kernels read them directly), else null
  int ld_sa;                   // leading dimension of the activation scales
  const int32_t* m_indices;    // contiguous: [M_total]
  const int32_t* masked_m;     // masked: [G]
  const int32_t* ks;           // K-grouped: [G] K rows of each group (multiples of 128)
  uint16_t* D;                 // bf16 output, [M][N] or [G][max_m][N]
  const uint16_t* C;           // dense / K-grouped: bf16 addend shaped like D (D = C + A B), or null
  unsigned int* status;        // device status word
  unsigned long long timeout_ns;
  unsigned int debug_flags;
};

}  // namespace dgk

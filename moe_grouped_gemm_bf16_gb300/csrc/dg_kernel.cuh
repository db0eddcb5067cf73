// The FP8 fine-grained-scaled GEMM kernel for sm_103a, written for GB300's
// tensor memory and TMA: the dense form, the contiguous and masked M-grouped
// forms and the K-grouped form, with the optional addend C.
//
// What it computes (DeepGEMM, es.news.hada.io/topic?id=19459, "Interfaz GEMM
// y restricciones de layout" and "Dense y Grouped GEMM"):
//   D[m,n] = bf16( C[m,n] + sum_g (A_g . B_g^T)[m,n] * sa[m,g] * sb[n/128,g] )
// with A e4m3 [M,K] and B e4m3 [N,K] (NT; the LAYOUT parameter also takes
// them stored [K,M] / [K,N]), one scale per row per 128-wide K group for A
// (stored K-group-major) and one per 128x128 block for B, fp32 or packed
// UE8M0 exponents.
//
// Structure (one persistent CTA per SM, a CTA pair, or one cluster of split_k
// CTAs per tile):
//   warps 0, 3  TMA producers (lane 0 of each, owning the ring slots of one
//               parity): A tile [128 x 128], B tile [BN x 128] into an
//               S-stage ring; the activation scales of four K groups at a
//               time into a separate ring (they are read later, by the
//               promotion warps); warp 0 also bulk-copies each tile's B
//               scales into one of two buffers, a tile ahead.
//   warps 1-2   warp 1 allocates tensor memory; the two warps take the K groups
//               in turn, one thread each issuing 4 tcgen05.mma (K = 32 each)
//               per K group into one of 2-4 TMEM accumulators, then
//               committing: the stage goes back to the producer, the
//               accumulator to the promotion warps.
//   warps 4..11 promotion (two warpgroups): read the group's fp32 partial from
//               TMEM, scale it by sa[m,g] * sb[n/128,g] and add it into fp32
//               registers while the tensor cores already compute the next
//               group (the two-level accumulation of the pages: DeepSeek's
//               overview deepep.org/zh/deepgemm, "细粒度缩放" / "核心优化技术").
//               Then the bf16 epilogue: a swizzled staging tile stored by TMA
//               (each promotion warp issuing some of the stores),
//               or, when the K groups are split over a cluster, a fixed-order
//               reduction of partials read through distributed shared memory.
//
// Every mbarrier wait is bounded: when one gives up it records a timeout in
// the device status word and sets a CTA-wide abort flag, after which every
// wait returns at once and no further TMA or MMA is issued, so the kernel runs
// to its normal end (all hardware barriers matched, TMEM freed) without
// hanging.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "dg_params.h"
#include "ptx.cuh"

namespace dgk {

// AROWS: rows of A loaded per tile (128, or 64 when M <= 64: the M=128 MMA
// then reads rows 64..127 of its A operand from the neighbouring slot, in
// bounds of the ring, and those output rows are discarded).
// PAIR: the CTA pair form (cta_group::2): each CTA holds half of the B tile.
template <int BN, int STAGES, bool SPLIT, int AROWS = BLOCK_M, bool PAIR = false>
struct SmemLayout {
  static constexpr int A_BYTES = AROWS * BLOCK_K;    // e4m3 A slot (16 KB or 8 KB)
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BLOCK_K;
  static constexpr int SA_BYTES = SA_GROUPS * BLOCK_M * 4;  // [SA_GROUPS][128] fp32
  // packed UE8M0 scales: the two words [2][128] that cover a slot's four K
  // groups wherever they start
  static constexpr int SA_PACKED_BYTES = 2 * BLOCK_M * 4;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int SA_OFF = B_OFF + STAGES * B_BYTES;
  // bf16 staging tile for the TMA store.  With the K split, each cluster
  // computes one tile, so after its last K group the operand ring is idle and
  // holds the fp32 partial of the reduction instead.
  static constexpr int OUT_OFF = SPLIT ? A_OFF : SA_OFF + SA_SLOTS * SA_BYTES;
  // split: the CTA's fp32 partial [AROWS][BN], which the cluster's owners read
  static constexpr int OUT_BYTES = SPLIT ? AROWS * BN * 4 : BLOCK_M * BN * 2;
  static_assert(!SPLIT || OUT_BYTES <= STAGES * (A_BYTES + B_BYTES), "partials must fit the ring");
  static constexpr int BAR_OFF = SPLIT ? SA_OFF + SA_SLOTS * SA_BYTES : OUT_OFF + OUT_BYTES;
  // barrier indexes
  static constexpr int FULL = 0, EMPTY = STAGES, SA_FULL = 2 * STAGES,
                       SA_EMPTY = 2 * STAGES + SA_SLOTS, T_FULL = 2 * STAGES + 2 * SA_SLOTS,
                       T_EMPTY = T_FULL + 4, READY = T_EMPTY + 4,
                       MMA_DONE = READY + 1, C_FULL = MMA_DONE + 1, SB_FULL = C_FULL + 1,
                       SB_EMPTY = SB_FULL + 2, NUM_BARS = SB_EMPTY + 2;
  // [0] TMEM base, [1] abort flag
  static constexpr int MISC_OFF = (BAR_OFF + NUM_BARS * 8 + 15) / 16 * 16;
  // checked build: fill counters of the operand ring's and the scale ring's slots
  static constexpr int DBG_OFF = MISC_OFF + 16;
  static constexpr int DBG_BYTES = kDebug ? ((STAGES + SA_SLOTS) * 4 + 15) / 16 * 16 : 0;
  // the B scale buffers (bulk-copy destinations: 16-byte aligned), then the
  // masked / K-grouped tables
  static constexpr int DYN_OFF = DBG_OFF + DBG_BYTES;
  static_assert(DYN_OFF % 16 == 0, "B scale buffers need 16-byte alignment");
  static_assert(B_OFF % 1024 == 0 && SA_OFF % 1024 == 0 && OUT_OFF % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  // TMEM accumulators (K groups the MMA may run ahead of the promotion warps):
  // as many BN-column buffers as the 512 columns hold, at most 4
  static constexpr int NBUF = (BN <= 128) ? 4 : 2;
  static constexpr int TMEM_COLS = (NBUF * BN <= 128) ? 128 : (NBUF * BN <= 256) ? 256 : 512;
};

// Dynamic shared memory a launch needs (host side too).
template <int BN, int STAGES, bool SPLIT, int AROWS = BLOCK_M, bool PAIR = false>
__host__ __device__ constexpr int smem_bytes(int kb, int num_groups, int mode) {
  return 1024 /* alignment slack */ + SmemLayout<BN, STAGES, SPLIT, AROWS, PAIR>::DYN_OFF +
         2 * sb_buf_words(kb) * 4 +
         (mode == kMasked ? (2 * num_groups + 1) * 4 : mode == kKGrouped ? (num_groups + 1) * 4 : 0);
}

struct Tile {
  int m0;     // first row of the tile, within its group
  int n0;     // first column
  int z;      // group coordinate of A / sa (masked form), else 0
  int zd;     // group coordinate of D / C (masked and K-grouped forms), else 0
  int e;      // expert / group of B and sb
  int rows;   // rows that hold valid output
  int skip;   // 1: contiguous padding block (no MMA, +0 output); 2: bad expert id;
              // 3: K-grouped group without K rows (no MMA, D = C or +0)
  int kbeg;   // the tile's K groups [kbeg, kend) (this CTA's slice in the split form)
  int kend;
};

// UE8M0 scale code -> fp32: 2^(e - 127) (e = 0: the subnormal 2^-127; 0xFF: NaN).
__device__ __forceinline__ float ue8m0_to_float(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u)
                : e == 0xFFu ? __uint_as_float(0x7FC00000u) : __uint_as_float(e << 23);
}

// Byte g % 4 of a packed UE8M0 word, as a scale.
__device__ __forceinline__ float ue8m0_scale(uint32_t word, int g) {
  return ue8m0_to_float((word >> (8 * (g & 3))) & 0xFFu);
}

__device__ __forceinline__ void raise_status(const Params& p, unsigned int code) {
  atomicCAS(p.status, 0u, code);
}

// Checked build: record a failed check and abort the CTA (every later wait
// returns at once and no further TMA or MMA is issued).
__device__ __forceinline__ void dbg_fail(const Params& p, unsigned int code,
                                         volatile uint32_t* abort_flag) {
  raise_status(p, code);
  *abort_flag = 1;
}

// Tile t of the persistent schedule.  Tiles are numbered in raster bands of
// `raster_m` M blocks: within a band, consecutive tiles walk down the band's M
// blocks and then across N, so the tiles running at the same time share A
// rows and B columns in L2 (block scheduler with rasterisation, DeepGEMM
// overview deepep.org/zh/deepgemm, "统一优化的块调度器").
// In the pair form an M block is 256 rows, of which CTA `crank` of the pair
// owns rows [128 * crank, 128 * crank + 128).
// K-grouped form: the tiles of group g come before those of g + 1 (each group
// rasterised alone); `prefix` holds the groups' first K groups.
// The contiguous form's expert id of the tile's first row is read from
// m_indices unless the caller passes it (pre_e >= -1, fetched ahead).
template <int BN, int MODE, bool PAIR = false>
__device__ __forceinline__ Tile decode_tile(int t, const Params& p, int num_m_blocks,
                                            const int* prefix, const int* mcnt, int kb0, int kb1,
                                            uint32_t crank = 0, int pre_e = -2) {
  const int nN = p.num_n_blocks;
  int kg = 0;
  if (MODE == kKGrouped) {
    const int per_group = num_m_blocks * nN;
    kg = t / per_group;
    t -= kg * per_group;
  }
  const int band_tiles = p.raster_m * nN;
  const int band = t / band_tiles;
  const int r = t - band * band_tiles;
  const int bm0 = band * p.raster_m;
  const int bh = min(p.raster_m, num_m_blocks - bm0);
  const int mb = bm0 + r % bh;
  Tile T;
  T.n0 = (r / bh) * BN;
  T.skip = 0;
  T.kbeg = kb0;
  T.kend = kb1;
  if (MODE == kKGrouped) {
    T.m0 = mb * BLOCK_M;
    T.z = 0;
    T.e = 0;
    T.rows = max(0, min(BLOCK_M, p.M - T.m0));
    T.kbeg = prefix[kg];
    T.kend = prefix[kg + 1];
    if (T.kend <= T.kbeg) T.skip = 3;
    T.zd = kg;
    return T;
  }
  if (MODE == kDense) {
    T.m0 = PAIR ? mb * 2 * BLOCK_M + static_cast<int>(crank) * BLOCK_M : mb * BLOCK_M;
    T.z = 0;
    T.e = 0;
    T.rows = max(0, min(BLOCK_M, p.M - T.m0));
  } else if (MODE == kContiguous) {
    T.m0 = mb * BLOCK_M;
    T.z = 0;
    const int e = pre_e >= -1 ? pre_e : __ldg(p.m_indices + T.m0);
    T.e = e;
    T.rows = BLOCK_M;
    if (e < 0) {
      T.skip = 1;
      T.e = 0;
    } else if (e >= p.num_groups) {
      T.skip = 2;
      T.e = 0;
    }
  } else {
    // flat M block -> group: largest g with prefix[g] <= mb
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= mb) lo = mid; else hi = mid - 1;
    }
    T.z = lo;
    T.e = lo;
    // pair form: M blocks of 256 rows, CTA `crank` owning 128 of them (the
    // second half may hold no valid row: it still takes part in the MMA and
    // stores nothing)
    T.m0 = PAIR ? (mb - prefix[lo]) * 2 * BLOCK_M + static_cast<int>(crank) * BLOCK_M
                : (mb - prefix[lo]) * BLOCK_M;
    T.rows = max(0, min(BLOCK_M, mcnt[lo] - T.m0));
  }
  T.zd = T.z;
  return T;
}

// First row of tile t in the contiguous form (decode_tile's raster order),
// so that its expert id can be fetched a tile ahead.
__device__ __forceinline__ int contiguous_tile_m0(int t, const Params& p, int num_m_blocks) {
  const int band_tiles = p.raster_m * p.num_n_blocks;
  const int band = t / band_tiles;
  const int r = t - band * band_tiles;
  const int bm0 = band * p.raster_m;
  const int bh = min(p.raster_m, num_m_blocks - bm0);
  return (bm0 + r % bh) * BLOCK_M;
}

// Checked build: the coordinates of a tile's loads for K group g lie inside
// the tensors (a pair's second half may start past M: its rows are zero-filled
// by design).
template <int MODE, bool PAIR>
__device__ __forceinline__ bool dbg_tile_ok(const Params& p, const Tile& T, int g) {
  const int zmax = MODE == kMasked ? p.num_groups : 1;
  const int emax = (MODE == kContiguous || MODE == kMasked) ? p.num_groups : 1;
  return g >= T.kbeg && g < T.kend && T.kbeg >= 0 && T.kend <= p.kb && T.m0 >= 0 &&
         T.m0 < p.M + (PAIR ? BLOCK_M : 0) && T.n0 >= 0 && T.n0 < p.N && T.z >= 0 && T.z < zmax &&
         T.e >= 0 && T.e < emax && T.zd >= 0 && T.zd < p.num_groups;
}

__device__ __forceinline__ int num_tiles_dense(const Params& p) {
  return p.num_m_blocks * p.num_n_blocks;
}

// Bounded mbarrier wait.  Returns false (without waiting) once the CTA has
// aborted, or after `timeout_ns`, in which case it records the timeout and
// aborts the CTA.
template <bool ACQ_CLUSTER = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         const Params& p) {
  auto try_once = [&]() {
    return ACQ_CLUSTER ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (try_once()) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (!try_once()) {
    if ((++it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        raise_status(p, ST_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
  return true;
}

// Wait used while draining at the end: ignores the abort flag, gives up only
// on the time limit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Params& p) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > p.timeout_ns) {
      raise_status(p, ST_TIMEOUT);
      return;
    }
  }
}

}  // namespace dgk

namespace dgk {

// SFP: the scales are packed UE8M0 exponents (a separate instance, so that the
// fp32-scale kernels carry no decode in their promotion loop).
template <int BN, int STAGES, bool SPLIT, int MODE, int AROWS = BLOCK_M, bool PAIR = false,
          int LAYOUT = kNT, bool SFP = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmD,
                const __grid_constant__ CUtensorMap tmC, const Params p) {
  static_assert(!SPLIT || MODE == kDense, "the K split is only used by the dense form");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN: multiple of 64 in [64, 256]");
  static_assert(AROWS == BLOCK_M || (AROWS == 64 && MODE == kDense), "64-row A: dense only");
  static_assert(!PAIR || (!SPLIT && (MODE == kDense || MODE == kMasked) && AROWS == BLOCK_M &&
                          (BN == 128 || BN == 256)),
                "the pair form: dense or masked, full A, 128- or 256-wide tiles");
  static_assert(LAYOUT == kNT || (!PAIR && AROWS == BLOCK_M && BN % 128 == 0 &&
                                   (MODE == kDense || MODE == kKGrouped)),
                "MN-major operands: dense (also K-split) or K-grouped, full A, 128-multiple tiles");
  static_assert(MODE != kKGrouped || LAYOUT == kTN, "the K-grouped form is tn");
  constexpr bool A_MN = (LAYOUT & 1) != 0;     // A stored [K][M]
  constexpr bool B_MN = (LAYOUT & 2) != 0;     // B stored [K][N]
  using L = SmemLayout<BN, STAGES, SPLIT, AROWS, PAIR>;
  constexpr int HALF = BN / PROMO_WG;          // columns per promotion warpgroup
  constexpr int NCH = HALF / 32;               // 32-column TMEM chunks per warpgroup
  // the pair MMA spans both CTAs' 128 rows
  constexpr uint32_t IDESC = idesc_e4m3_f32(PAIR ? 2 * BLOCK_M : BLOCK_M, BN, A_MN, B_MN);
  // An MN-major operand slot holds 128 K rows of 128-byte lines per 128-wide
  // atom (16 KB each, stacked along M / N); the MMA's K step of 32 is then 4
  // swizzle atoms (4096 bytes) further on, against 32 bytes inside the atom
  // for a K-major slot.
  constexpr uint32_t MN_ATOM_BYTES = 128 * BLOCK_K;
  constexpr uint64_t A_KSTEP = A_MN ? (32 * 128) >> 4 : 32 >> 4;
  constexpr uint64_t B_KSTEP = B_MN ? (32 * 128) >> 4 : 32 >> 4;

  extern __shared__ uint8_t smem_raw[];
  // swizzled tiles need 1024-byte aligned shared-memory addresses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8 * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile uint32_t* abort_flag = misc + 1;
  // B scales of a tile, two buffers (one filled while the other is read)
  float* sb_s = reinterpret_cast<float*>(smem + L::DYN_OFF);
  const int sbw = sb_buf_words(p.kb);
  int* prefix = reinterpret_cast<int*>(sb_s + 2 * sbw);
  int* mcnt = prefix + p.num_groups + 1;
  const float* sa_ring = reinterpret_cast<const float*>(smem + L::SA_OFF);
  // checked build: fills of each operand-ring slot, then of each scale-ring slot
  volatile uint32_t* dbg_fill = reinterpret_cast<volatile uint32_t*>(smem + L::DBG_OFF);
  volatile uint32_t* dbg_sa_fill = dbg_fill + STAGES;

  const uint32_t crank = (SPLIT || PAIR) ? cluster_ctarank() : 0;
  const int S = SPLIT ? p.split_k : 1;           // CTAs sharing one tile's K groups
  const int CL = PAIR ? 2 : S;                   // CTAs per cluster
  const bool leader = crank == 0;                // pair form: the CTA that issues the MMAs
  const int cluster_id = blockIdx.x / CL;
  const int num_clusters = gridDim.x / CL;
  // this CTA's K groups: a slice of them in the split form, all of them otherwise
  // (the pair form's cluster rank names a half of the tile, not of K)
  const uint32_t krank = SPLIT ? crank : 0;
  // A tile's B scales come either from the producer or from the promotion
  // threads' own 4-byte copies (the K split, whose CTAs take a slice of each
  // row, and the K-grouped form, whose rows are per group).  The producer
  // copies, in one bulk copy, the 16-byte aligned span of global memory that
  // holds the rows of the tile's 128-column blocks (consecutive rows of the
  // scale tensor); a row starts `sb_lead` words into the span.  Either way
  // they land in one of two buffers while the previous tile is promoted.
  const bool sb_bulk = !SPLIT && MODE != kKGrouped;
  const int sb_row = SFP ? p.kbp : p.kb;   // words per row of the scale tensor
  auto sb_first_row = [&](const Tile& U) {
    return reinterpret_cast<const uint32_t*>(p.sb) +
           (static_cast<size_t>(U.e) * p.nb + (U.n0 >> 7)) * sb_row;
  };
  const int kbeg = static_cast<int>(static_cast<long long>(krank) * p.kb / S);
  const int kend = static_cast<int>(static_cast<long long>(krank + 1) * p.kb / S);

  // ------------------------------------------------------------- set-up --
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(L::FULL + s), 1);
      mbar_init(bar(L::EMPTY + s), 1);
    }
    for (int j = 0; j < SA_SLOTS; ++j) {
      mbar_init(bar(L::SA_FULL + j), 1);
      mbar_init(bar(L::SA_EMPTY + j), NUM_PROMO_WARPS);
    }
    for (int b = 0; b < L::NBUF; ++b) {
      mbar_init(bar(L::T_FULL + b), 1);
      // pair form: the leader's barrier counts both CTAs' promotion warps
      mbar_init(bar(L::T_EMPTY + b), PAIR ? 2 * NUM_PROMO_WARPS : NUM_PROMO_WARPS);
    }
    mbar_init(bar(L::READY), S);
    mbar_init(bar(L::MMA_DONE), NUM_ISSUERS);
    mbar_init(bar(L::C_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::SB_FULL + i), sb_bulk ? 1 : 32 * NUM_PROMO_WARPS);
      mbar_init(bar(L::SB_EMPTY + i), NUM_PROMO_WARPS);
    }
    misc[1] = 0;
    if constexpr (kDebug)
      for (int i = 0; i < STAGES + SA_SLOTS; ++i) dbg_fill[i] = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSA);
    prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(sbase + L::MISC_OFF, L::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(sbase + L::MISC_OFF, L::TMEM_COLS);
      tmem_relinquish();
    }
  }
  // Dense nt form: ask L2 for the B boxes of this CTA's first two K groups
  // while the previous kernel in the stream may still run (a CTA that starts
  // early, on an SM that kernel left free, would otherwise only wait).  A
  // prefetch delivers nothing to this CTA and L2 is where all writes meet, so
  // it cannot hand out stale data even if the previous kernel writes B; the
  // loads themselves still come after the wait below.  (A cold first load
  // measured 2-3 us after the wait in back-to-back decode GEMMs.)
  if (MODE == kDense && LAYOUT == kNT && !PAIR && warp == 0 && lane == 0 &&
      cluster_id < p.num_m_blocks * p.num_n_blocks) {
    const Tile T0 = decode_tile<BN, MODE, PAIR>(cluster_id, p, p.num_m_blocks, nullptr, nullptr,
                                                kbeg, kend, crank);
    for (int g = T0.kbeg; g < T0.kend && g < T0.kbeg + 2; ++g)
      tma_prefetch_3d(&tmB, g * BLOCK_K, T0.n0, T0.e);
  }
  // Everything above touched only shared memory, tensor memory and the kernel
  // parameters (and asked L2 for B, above); global memory (which the previous
  // kernel in the stream may still be writing) is read only after this wait.
  // Dependent launches may start their own prologue from here on.
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (MODE == kMasked && warp == 2) {  // (warp 2 has no other set-up work)
    // valid rows per group (clamped to [0, max_m]) and the prefix sum of M blocks
    int carry = 0;
    for (int base = 0; base < p.num_groups; base += 32) {
      const int g = base + lane;
      int c = 0;
      if (g < p.num_groups) {
        const int v = __ldg(p.masked_m + g);
        const int vc = min(max(v, 0), p.M);
        if (vc != v && blockIdx.x == 0) raise_status(p, ST_MASK_RANGE);
        mcnt[g] = vc;
        c = PAIR ? (vc + 2 * BLOCK_M - 1) / (2 * BLOCK_M) : (vc + BLOCK_M - 1) / BLOCK_M;
      }
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (g < p.num_groups) prefix[g + 1] = carry + x;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  if (MODE == kKGrouped && warp == 2) {
    // first K group of every group: prefix sum of ks[g] / 128, each ks[g]
    // checked (>= 0, whole K groups) and the running total clamped to K
    int carry = 0;
    bool bad = false;
    for (int base = 0; base < p.num_groups; base += 32) {
      const int g = base + lane;
      int c = 0;
      if (g < p.num_groups) {
        const int v = __ldg(p.ks + g);
        if (v < 0 || (v & (BLOCK_K - 1)) != 0) bad = true;
        c = max(v, 0) / BLOCK_K;
      }
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (g < p.num_groups) {
        if (carry + x > p.kb) bad = true;
        prefix[g + 1] = min(carry + x, p.kb);
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
      carry = min(carry, p.kb);
    }
    if (lane == 0) prefix[0] = 0;
    if (bad && blockIdx.x == 0) raise_status(p, ST_KS_RANGE);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // peers signal this CTA's barriers from here on: thread 0 made their
  // initialisation visible to the cluster (fence.mbarrier_init), so a relaxed
  // rendezvous suffices
  if (SPLIT || PAIR) {
    cluster_arrive_relaxed();
    cluster_wait();
  }
  const uint32_t tmem_base = misc[0];
  const int num_m_blocks = (MODE == kMasked) ? prefix[p.num_groups] : p.num_m_blocks;
  const int num_tiles =
      num_m_blocks * p.num_n_blocks * (MODE == kKGrouped ? p.num_groups : 1);
  // the split form computes exactly one tile per cluster (the host launches one
  // cluster per tile); the operand ring is reused by its epilogue
  const int tile_stride = SPLIT ? num_tiles : num_clusters;

  // Move registers from warpgroup 0 (TMA, MMA issue, an idle warp) to the
  // promotion warpgroups when their accumulators need them.  The shares add up
  // to what the launch holds: two promotion warpgroups (384 threads, 168 each):
  // 40 + 2 * 232 = 3 * 168; four (640 threads, 96 each): 32 + 4 * 112 = 5 * 96.
  constexpr bool REALLOC = PROMO_WG == 4 || HALF >= 128;
  constexpr uint32_t REGS_CTRL = PROMO_WG == 4 ? 32 : 40;
  constexpr uint32_t REGS_PROMO = PROMO_WG == 4 ? 112 : 232;
  static_assert(REGS_CTRL + PROMO_WG * REGS_PROMO <= (1 + PROMO_WG) * (PROMO_WG == 4 ? 96 : 168),
                "register shares exceed the launch's registers");

  if (warp < 4) {
  if constexpr (REALLOC) regs_dec<REGS_CTRL>();
  if (warp == 0 || warp == 3) {
    // ----------------------------------------------------- TMA producers --
    // Two threads (warps 0 and 3) share the loads: a thread that issues a TMA
    // load stalls for ~250 cycles, so one thread issuing every K group's
    // loads falls behind the MMA.  Each owns fixed slots (operand stages and
    // activation-scale slots of its parity), so every slot's latest fill is
    // its owner's, which the drain below relies on.  Both walk the whole
    // sequence, so their ring positions agree.
    if (lane == 0 && !(p.debug_flags & DBG_SKIP_PRODUCER)) {
      const int me = warp == 3 ? 1 : 0;
      // per slot: was a load issued, and with which phase parity
      uint32_t issued_mask = 0, issued_par = 0, sa_issued_mask = 0, sa_issued_par = 0;
      int s = 0, j = 0;
      uint32_t ph = 0, jph = 0;
      uint32_t sbb = 0, sb_eph = 0, sb_issued = 0, sb_par = 0;   // B scale buffers (bulk form)
      for (int t = cluster_id; t < num_tiles; t += tile_stride) {
        const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, kbeg, kend, crank);
        if (sb_bulk && me == 0) {
          // the tile's B scales: rows of the (up to 3) 128-column blocks, once
          // the promotion threads are done with the buffer's previous tile
          if (wait_bar(bar(L::SB_EMPTY + sbb), ((sb_eph >> sbb) & 1u) ^ 1u, abort_flag, p)) {
            // (the drain below waits for the buffer's latest phase, which a
            // padding tile's plain arrival completes as well)
            sb_issued |= 1u << sbb;
            sb_par = (sb_par & ~(1u << sbb)) | (((sb_eph >> sbb) & 1u) << sbb);
            if (T.skip) {
              mbar_arrive(bar(L::SB_FULL + sbb));
            } else {
              // the rows of the blocks the tile's columns touch, within N (the
              // buffer's rows past them are never read for a stored column);
              // the span is widened to 16-byte boundaries, which never leaves
              // the memory pages of the rows themselves
              const int nrows = min(((T.n0 & 127) + BN - 1) / 128 + 1, p.nb - (T.n0 >> 7));
              const uintptr_t a = reinterpret_cast<uintptr_t>(sb_first_row(T));
              const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
              const uintptr_t a1 = (a + static_cast<uintptr_t>(nrows) * sb_row * 4u + 15) &
                                   ~static_cast<uintptr_t>(15);
              const uint32_t bytes = static_cast<uint32_t>(a1 - a0);
              mbar_arrive_expect_tx(bar(L::SB_FULL + sbb), bytes);
              bulk_load_g2s(smem_u32(sb_s + sbb * sbw), reinterpret_cast<const void*>(a0), bytes,
                            bar(L::SB_FULL + sbb));
            }
          }
          sb_eph ^= 1u << sbb;
          sbb ^= 1u;
        }
        if (T.skip) continue;
        for (int g = T.kbeg; g < T.kend; ++g) {
          if ((s & 1) != me) {   // the other producer's stage
            if ((g - T.kbeg) % SA_GROUPS == 0) {
              if ((j & 1) == me) {
                // this producer's scale slot, on the other's group
                bool sgo = wait_bar(bar(L::SA_EMPTY + j), jph ^ 1, abort_flag, p);
                if constexpr (kDebug) {
                  if (sgo && (g < 0 || (SFP ? (g >> 2) >= p.kbp : g >= p.kb))) {
                    dbg_fail(p, ST_DEBUG_BOUNDS, abort_flag);
                    sgo = false;
                  }
                  if (sgo) dbg_sa_fill[j] = dbg_sa_fill[j] + 1;
                }
                if (sgo) {
                  if constexpr (SFP) {
                    mbar_arrive_expect_tx(bar(L::SA_FULL + j), L::SA_PACKED_BYTES);
                    tma_load_3d(sbase + L::SA_OFF + j * L::SA_BYTES, &tmSA, bar(L::SA_FULL + j),
                                T.m0, g >> 2, T.z);
                  } else {
                    mbar_arrive_expect_tx(bar(L::SA_FULL + j), L::SA_BYTES);
                    tma_load_3d(sbase + L::SA_OFF + j * L::SA_BYTES, &tmSA, bar(L::SA_FULL + j),
                                T.m0, g, T.z);
                  }
                  sa_issued_mask |= 1u << j;
                  sa_issued_par = (sa_issued_par & ~(1u << j)) | (jph << j);
                }
              }
              if (++j == SA_SLOTS) { j = 0; jph ^= 1; }
            }
            if (++s == STAGES) { s = 0; ph ^= 1; }
            continue;
          }
          bool go = wait_bar(bar(L::EMPTY + s), ph ^ 1, abort_flag, p);
          if constexpr (kDebug) {
            if (go && !dbg_tile_ok<MODE, PAIR>(p, T, g)) {
              dbg_fail(p, ST_DEBUG_BOUNDS, abort_flag);
              go = false;
            }
            if (go) dbg_fill[s] = dbg_fill[s] + 1;
          }
          if (go) {
            if constexpr (PAIR) {
              // both CTAs' loads complete on the leader's FULL barrier, which
              // expects the bytes of both
              // (destinations as cluster addresses of this CTA's own shared memory)
              const uint32_t full = map_cluster(bar(L::FULL + s), 0);
              if (leader) mbar_arrive_expect_tx(bar(L::FULL + s), 2 * (L::A_BYTES + L::B_BYTES));
              tma_load_3d_pair(map_cluster(sbase + L::A_OFF + s * L::A_BYTES, crank), &tmA, full,
                               g * BLOCK_K, T.m0, T.z);
              tma_load_3d_pair(map_cluster(sbase + L::B_OFF + s * L::B_BYTES, crank), &tmB, full,
                               g * BLOCK_K, T.n0 + static_cast<int>(crank) * (BN / 2), T.e);
            } else if constexpr (LAYOUT != kNT) {
              // MN-major operands: boxes of 128 (M or N) x 128 K rows; an
              // MN-major B's boxes wholly past N are not loaded (their columns
              // are never stored).  A K-major B is one full box as in nt.
              int nbox = 0;
              for (int bj = 0; bj < BN / 128; ++bj) nbox += (T.n0 + bj * 128 < p.N) ? 1 : 0;
              const uint32_t b_bytes = B_MN ? nbox * MN_ATOM_BYTES : L::B_BYTES;
              mbar_arrive_expect_tx(bar(L::FULL + s), L::A_BYTES + b_bytes);
              const uint32_t a_dst = sbase + L::A_OFF + s * L::A_BYTES;
              const uint32_t b_dst = sbase + L::B_OFF + s * L::B_BYTES;
              if constexpr (A_MN)
                tma_load_3d(a_dst, &tmA, bar(L::FULL + s), T.m0, g * BLOCK_K, T.z);
              else
                tma_load_3d(a_dst, &tmA, bar(L::FULL + s), g * BLOCK_K, T.m0, T.z);
              if constexpr (B_MN) {
                for (int bj = 0; bj < nbox; ++bj)
                  tma_load_3d(b_dst + bj * MN_ATOM_BYTES, &tmB, bar(L::FULL + s), T.n0 + bj * 128,
                              g * BLOCK_K, T.e);
              } else {
                tma_load_3d(b_dst, &tmB, bar(L::FULL + s), g * BLOCK_K, T.n0, T.e);
              }
            } else {
              mbar_arrive_expect_tx(bar(L::FULL + s), L::A_BYTES + L::B_BYTES);
              tma_load_3d(sbase + L::A_OFF + s * L::A_BYTES, &tmA, bar(L::FULL + s), g * BLOCK_K,
                          T.m0, T.z);
              tma_load_3d(sbase + L::B_OFF + s * L::B_BYTES, &tmB, bar(L::FULL + s), g * BLOCK_K,
                          T.n0, T.e);
            }
            issued_mask |= 1u << s;
            issued_par = (issued_par & ~(1u << s)) | (ph << s);
          }
          // the scales of this and the next SA_GROUPS-1 K groups (groups past
          // the tensor's end read as zero and are not used), if the slot is
          // this producer's
          if ((g - T.kbeg) % SA_GROUPS == 0 && (j & 1) != me) {
            if (++j == SA_SLOTS) { j = 0; jph ^= 1; }
          } else if ((g - T.kbeg) % SA_GROUPS == 0) {
            bool sgo = wait_bar(bar(L::SA_EMPTY + j), jph ^ 1, abort_flag, p);
            if constexpr (kDebug) {
              if (sgo && (g < 0 || (SFP ? (g >> 2) >= p.kbp : g >= p.kb))) {
                dbg_fail(p, ST_DEBUG_BOUNDS, abort_flag);
                sgo = false;
              }
              if (sgo) dbg_sa_fill[j] = dbg_sa_fill[j] + 1;
            }
            if (sgo) {
              if constexpr (SFP) {
                mbar_arrive_expect_tx(bar(L::SA_FULL + j), L::SA_PACKED_BYTES);
                tma_load_3d(sbase + L::SA_OFF + j * L::SA_BYTES, &tmSA, bar(L::SA_FULL + j), T.m0,
                            g >> 2, T.z);
              } else {
                mbar_arrive_expect_tx(bar(L::SA_FULL + j), L::SA_BYTES);
                tma_load_3d(sbase + L::SA_OFF + j * L::SA_BYTES, &tmSA, bar(L::SA_FULL + j), T.m0,
                            g, T.z);
              }
              sa_issued_mask |= 1u << j;
              sa_issued_par = (sa_issued_par & ~(1u << j)) | (jph << j);
            }
            if (++j == SA_SLOTS) { j = 0; jph ^= 1; }
          }
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
      }
      // Drain: after an abort the latest load into a slot may still be in
      // flight; wait for it before the CTA can exit.  (After a normal run every
      // load has been consumed already and these waits return at once.)
      // (pair form: the leader's FULL barriers count both CTAs' loads, and the
      // leader drains them; the CTAs leave only together, after a rendezvous)
      for (int q = 0; q < STAGES; ++q)
        if (((issued_mask >> q) & 1u) && (!PAIR || leader))
          drain_wait(bar(L::FULL + q), (issued_par >> q) & 1u, p);
      for (int q = 0; q < SA_SLOTS; ++q)
        if ((sa_issued_mask >> q) & 1u) drain_wait(bar(L::SA_FULL + q), (sa_issued_par >> q) & 1u, p);
      for (int q = 0; q < 2; ++q)
        if ((sb_issued >> q) & 1u) drain_wait(bar(L::SB_FULL + q), (sb_par >> q) & 1u, p);
    }
    __syncwarp();
  } else if (warp <= NUM_ISSUERS) {
    // ------------------------------------------------------ MMA issuers ---
    // A thread that issues tcgen05.mma stalls until the tensor pipe takes the
    // instruction, so the barrier waits between one K group's MMAs and the
    // next would leave the pipe idle.  Warps 1..NUM_ISSUERS take the K groups
    // in turn: while one waits for its stage and accumulator, another's MMAs
    // run.  Group g goes to issuer g mod NUM_ISSUERS.
    // The parity waits stay exact: (1) NUM_ISSUERS divides NBUF, so the issuer
    // of group g also issued group g - NBUF on the same accumulator buffer and
    // saw its release phase before, which rules out a barrier two phases behind;
    // (2) STAGES >= NBUF, so once the accumulator of g - NBUF is released (the
    // promotion runs in group order) the MMAs of every group up to g - NBUF,
    // g - STAGES among them, have completed, and the stage's previous fill
    // phase is over.  With an issuer count that does not divide NBUF a wait can
    // pass a phase early and the barrier accounting breaks down.
    // (pair form: the leader issues for both CTAs; the other CTA's warp 1 only
    // takes part in the collective TMEM allocation)
    static_assert(L::NBUF % NUM_ISSUERS == 0 && STAGES >= L::NBUF,
                  "issuer turns must keep every barrier within one phase");
    if (lane == 0 && (!PAIR || leader)) {
      const int me = warp - 1;
      int s = 0, b = 0, turn = 0;
      uint32_t ph = 0, bph = 0;
      uint32_t q = 0;   // K groups of this CTA's sequence so far (both issuers' turns)
      for (int t = cluster_id; t < num_tiles; t += tile_stride) {
        const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, kbeg, kend, crank);
        if (T.skip) continue;
        for (int g = T.kbeg; g < T.kend; ++g, ++q) {
          const bool mine = (turn == me);
          if (++turn == NUM_ISSUERS) turn = 0;
          if (!mine) {
            if (++s == STAGES) { s = 0; ph ^= 1; }
            if (++b == L::NBUF) { b = 0; bph ^= 1; }
            continue;
          }
          const bool ok_t = wait_bar(bar(L::T_EMPTY + b), bph ^ 1, abort_flag, p);
          tc_fence_after();
          bool ok_f = wait_bar(bar(L::FULL + s), ph, abort_flag, p);
          tc_fence_after();
          if constexpr (kDebug) {
            // the stage holds this group's fill: its (q / STAGES + 1)-th
            if (ok_f && dbg_fill[s] != q / STAGES + 1) {
              dbg_fail(p, ST_DEBUG_PHASE, abort_flag);
              ok_f = false;
            }
          }
          if (ok_t && ok_f) {
            const uint32_t d = tmem_base + static_cast<uint32_t>(b * BN);
            const uint32_t a_src = sbase + L::A_OFF + s * L::A_BYTES;
            const uint32_t b_src = sbase + L::B_OFF + s * L::B_BYTES;
            const uint64_t ad = A_MN ? smem_desc_sw128_mnmajor(a_src, MN_ATOM_BYTES)
                                     : smem_desc_sw128_kmajor(a_src);
            const uint64_t bd = B_MN ? smem_desc_sw128_mnmajor(b_src, MN_ATOM_BYTES)
                                     : smem_desc_sw128_kmajor(b_src);
            if constexpr (PAIR) {
#pragma unroll
              for (int kk = 0; kk < BLOCK_K / 32; ++kk)
                mma_f8f6f4_pair(d, ad + A_KSTEP * kk, bd + B_KSTEP * kk, IDESC, kk > 0 ? 1u : 0u);
              // frees the stage and hands the accumulator over in both CTAs
              mma_commit_pair_multicast(bar(L::EMPTY + s), 0x3);
              mma_commit_pair_multicast(bar(L::T_FULL + b), 0x3);
            } else {
#pragma unroll
              for (int kk = 0; kk < BLOCK_K / 32; ++kk)
                mma_f8f6f4(d, ad + A_KSTEP * kk, bd + B_KSTEP * kk, IDESC, kk > 0 ? 1u : 0u);
              mma_commit(bar(L::EMPTY + s));
              mma_commit(bar(L::T_FULL + b));
            }
          }
          if (++s == STAGES) { s = 0; ph ^= 1; }
          if (++b == L::NBUF) { b = 0; bph ^= 1; }
        }
      }
      // nothing issued may still run when the TMEM is freed
      if constexpr (PAIR) mma_commit_pair_multicast(bar(L::MMA_DONE), 0x1);
      else mma_commit(bar(L::MMA_DONE));
      drain_wait(bar(L::MMA_DONE), 0, p);
    }
    __syncwarp();
  }
  } else {
    if constexpr (REALLOC) regs_inc<REGS_PROMO>();
    // -------------------------------------------------- promotion warps ---
    const int pw = warp - 4;            // 0 .. NUM_PROMO_WARPS-1
    const int q = warp & 3;             // TMEM lane quadrant this warp may access
    const int h = pw >> 2;              // which column share of the tile
    const int row = q * 32 + lane;      // the tile row this thread owns
    const int pt = threadIdx.x - 128;   // index among the promotion threads
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t out_s = sbase + L::OUT_OFF;
    int b = 0, j = 0;
    uint32_t bph = 0, jph = 0;
    uint32_t jn = 0;                    // scale-ring slots consumed (checked build)
    uint32_t k_iter = 0;                // tiles finished (phase of the reduction barriers)
    uint32_t cph = 0;                   // phase of the addend's barrier
    float acc[HALF];
    // B scales: a tile's scale i (i < 3 * its K groups) is 128-column block
    // i / groups, K group i % groups (packed form: the word holding that
    // group's byte, decoded where it is read).  They are copied (cp.async, 4
    // bytes each) into one of two buffers while the previous tile is
    // promoted, completing on that buffer's mbarrier (one arrival per
    // promotion thread, signalled after the tile's last K group: the arrival
    // instruction held the issuing warp until its copies had landed); a load
    // issued at the tile's start would hold up its first promotion by the
    // load's latency.
    auto sb_issue = [&](int tt, uint32_t buf) {
      if (sb_bulk) return;
      const Tile U = decode_tile<BN, MODE, PAIR>(tt, p, num_m_blocks, prefix, mcnt, kbeg, kend, crank);
      if (!U.skip) {
        const int tku = U.kend - U.kbeg;
        float* dst = sb_s + buf * sbw;
        for (int i = pt; i < 3 * tku; i += 32 * NUM_PROMO_WARPS) {
          const int jb = i / tku, gg = i - jb * tku;
          const int nbk = min((U.n0 >> 7) + jb, p.nb - 1);
          const void* src;
          if constexpr (SFP)
            src = reinterpret_cast<const uint32_t*>(p.sb) +
                  (static_cast<size_t>(U.e) * p.nb + nbk) * p.kbp + ((U.kbeg + gg) >> 2);
          else
            src = p.sb + (static_cast<size_t>(U.e) * p.nb + nbk) * p.kb + U.kbeg + gg;
          cp_async_4(smem_u32(dst + i), src);
        }
      }
    };
    uint32_t sbi = 0;                   // buffer of the current tile's B scales
    uint32_t sbph = 0;                  // phase bit of each buffer's barrier
    if (cluster_id < num_tiles && !sb_bulk) {
      sb_issue(cluster_id, 0);
      cp_async_mbar_arrive_noinc(bar(L::SB_FULL + 0));
    }
    // contiguous form: the expert id of the next tile's first row, and each
    // row's id for this tile's epilogue, are loaded a tile / a main loop
    // ahead (each load is a round trip to memory that would otherwise stall
    // the promotion warps at the tile's start and at its epilogue)
    int e_next = (MODE == kContiguous && cluster_id < num_tiles)
                     ? __ldg(p.m_indices + contiguous_tile_m0(cluster_id, p, num_m_blocks))
                     : -2;
    for (int t = cluster_id; t < num_tiles; t += tile_stride, ++k_iter) {
      const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, kbeg, kend, crank,
                                                 MODE == kContiguous ? e_next : -2);
      int row_id = -1;
      if constexpr (MODE == kContiguous) {
        if (!T.skip) row_id = __ldg(p.m_indices + T.m0 + row);
        if (t + tile_stride < num_tiles)
          e_next = __ldg(p.m_indices + contiguous_tile_m0(t + tile_stride, p, num_m_blocks));
      }
      // Dense form with an addend (D = C + A B^T): thread 0 loads this tile's C
      // into the staging tile, in the store's own layout, halfway through the
      // tile's K groups (the previous tile's store has long finished reading
      // the staging tile by then, and C has long landed by the epilogue).
      const bool load_c = (MODE == kDense || MODE == kKGrouped) && !SPLIT && p.C != nullptr && pt == 0;
      const int tk = T.kend - T.kbeg;     // the tile's K groups
      const int g_c = (T.skip || tk <= 0) ? -1 : T.kbeg + tk / 2;   // K group after which C loads
      auto issue_c = [&]() {
        bulk_wait_group_read0();
        uint32_t bytes = 0;
        for (int cc = 0; cc < BN / 32; ++cc)
          if (T.n0 + cc * 32 < p.N) bytes += BLOCK_M * 64;
        mbar_arrive_expect_tx(bar(L::C_FULL), bytes);
        for (int cc = 0; cc < BN / 32; ++cc)
          if (T.n0 + cc * 32 < p.N)
            tma_load_3d(out_s + cc * (BLOCK_M * 64), &tmC, bar(L::C_FULL), T.n0 + cc * 32, T.m0,
                        T.zd);
      };
      // this tile's B scales (every promotion thread's copies have landed);
      // the other buffer, last read by the previous tile, which every thread
      // has finished, takes the next tile's
      // (bulk form: the tile's first row starts a few words into the span)
      const float* sbt =
          sb_s + sbi * sbw +
          ((sb_bulk && !T.skip) ? (reinterpret_cast<uintptr_t>(sb_first_row(T)) >> 2) & 3 : 0);
      // words between the rows of consecutive 128-column blocks
      const int rstride = sb_bulk ? sb_row : tk;
      wait_bar(bar(L::SB_FULL + sbi), (sbph >> sbi) & 1u, abort_flag, p);
      sbph ^= 1u << sbi;
      const bool sb_next = t + tile_stride < num_tiles;
      if (sb_next) sb_issue(t + tile_stride, sbi ^ 1u);
      sbi ^= 1u;
      if ((MODE == kDense || MODE == kKGrouped) && !SPLIT && p.C != nullptr) {
        // with an addend, the staging tile receives C during this tile: every
        // store of the previous tile (several warps issue them, each waiting
        // for its own) must have read it first
        if (lane == 0) bulk_wait_group_read0();
        named_bar_sync(1, 32 * NUM_PROMO_WARPS);
        if (load_c && g_c < 0) issue_c();
      }
#pragma unroll
      for (int i = 0; i < HALF; ++i) acc[i] = 0.f;
      if (!T.skip) {
        const int nmod = T.n0 & 127;
        for (int g = T.kbeg; g < T.kend; ++g) {
          // hand the TMEM accumulator back to the MMA issuer (pair form: on the
          // leader's barrier); every tcgen05.ld of this warp has completed
          auto release_tmem = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (PAIR && !leader) mbar_arrive_remote_relaxed(bar(L::T_EMPTY + b), 0);
              else mbar_arrive(bar(L::T_EMPTY + b));
            }
          };
          const int r = (g - T.kbeg) % SA_GROUPS;   // place in the scale slot
          wait_bar(bar(L::T_FULL + b), bph, abort_flag, p);
          if (r == 0) {
            const bool ok_sa = wait_bar(bar(L::SA_FULL + j), jph, abort_flag, p);
            if constexpr (kDebug) {
              if (ok_sa && dbg_sa_fill[j] != jn / SA_SLOTS + 1) dbg_fail(p, ST_DEBUG_PHASE, abort_flag);
            }
          }
          __syncwarp();
          tc_fence_after();
          // warps whose TMEM lanes hold no loaded row of A have nothing to add
          if (q * 32 < AROWS) {
          // packed: word (g/4 - first group/4) of the slot, byte g % 4
          float a_s;
          if constexpr (SFP)
            a_s = ue8m0_scale(reinterpret_cast<const uint32_t*>(
                                  sa_ring)[(j * SA_GROUPS + ((g >> 2) - ((g - r) >> 2))) *
                                               BLOCK_M + row], g);
          else
            a_s = sa_ring[(j * SA_GROUPS + r) * BLOCK_M + row];
          // bulk form, packed scales: one word per four K groups
          const float* sbg = sbt + ((sb_bulk && SFP) ? (g >> 2) : (g - T.kbeg));
          const uint32_t tcol = t_lane + static_cast<uint32_t>(b * BN + h * HALF);
          // PROMO_LB 32-column chunks per load batch: tcgen05.wait::ld waits for
          // every outstanding load, so fewer, larger batches expose its latency
          // fewer times.  The accumulator is released as soon as the last batch
          // is in registers, before that batch is scaled and added.
          constexpr int LB = NCH < PROMO_LB ? NCH : PROMO_LB;
          constexpr int NB = NCH / LB;
          static_assert(NCH % LB == 0, "whole load batches");
#pragma unroll
          for (int bt = 0; bt < NB; ++bt) {
            uint32_t v[LB][32];
#pragma unroll
            for (int u = 0; u < LB; ++u)
              tmem_ld_32x32b_x32(tcol + (bt * LB + u) * 32, v[u]);
#pragma unroll
            for (int u = 0; u < LB; ++u) tmem_wait_ld(v[u]);
            if (bt == NB - 1) release_tmem();
#pragma unroll
            for (int u = 0; u < LB; ++u) {
              const int c = bt * LB + u;
              const int col = h * HALF + c * 32;
              // the 32 columns lie in one 128-column B scale block
              const float sb_v = sbg[((nmod + col) >> 7) * rstride];
              const float sc = a_s * (SFP ? ue8m0_scale(__float_as_uint(sb_v), g) : sb_v);
#pragma unroll
              for (int i = 0; i < 32; i += 2)
                ffma2(acc[c * 32 + i], acc[c * 32 + i + 1], __uint_as_float(v[u][i]),
                      __uint_as_float(v[u][i + 1]), sc);
            }
          }
          } else {
            release_tmem();
          }
          if (r == SA_GROUPS - 1 || g == T.kend - 1) {
            // the slot's last K group of this tile: hand the slot back
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::SA_EMPTY + j));
            if (++j == SA_SLOTS) { j = 0; jph ^= 1; }
            ++jn;
          }
          if (++b == L::NBUF) { b = 0; bph ^= 1; }
          if (load_c && g == g_c) issue_c();
        }
      }
      if (sb_bulk) {
        // (this tile's buffer is the other one now)
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::SB_EMPTY + (sbi ^ 1u)));
      } else if (sb_next) {
        cp_async_mbar_arrive_noinc(bar(L::SB_FULL + sbi));
      }
      if constexpr (!SPLIT) {
        // ------------------------------------ epilogue: bf16 via TMA store --
        bool zero_row = false;  // contiguous form: padding rows (m_indices = -1) are +0
        if constexpr (MODE == kContiguous) {
          if (T.skip) {
            zero_row = true;
            if (T.skip == 2 && pt == 0) raise_status(p, ST_EXPERT_RANGE);
          } else {
            const int id = row_id;
            if (id != T.e) {
              zero_row = true;
              if (id >= 0) raise_status(p, ST_EXPERT_RANGE);  // block mixes two experts
            }
          }
        }
        // dense form with an addend: wait for this tile's C in the staging tile
        // (each thread reads exactly the 16-byte units it writes below)
        bool c_in = false;
        if constexpr (MODE == kDense || MODE == kKGrouped) {
          if (p.C != nullptr) {
            c_in = wait_bar(bar(L::C_FULL), cph, abort_flag, p);
            cph ^= 1;
          }
        }
        // the previous tile's stores (one or more per warp) have read the staging tile
        if (lane == 0) bulk_wait_group_read0();
        named_bar_sync(1, 32 * NUM_PROMO_WARPS);
        // staging: BN/32 chunks of [128 rows x 64 B], 64-byte swizzle (16-byte
        // unit u of row r sits at unit u ^ ((r >> 1) & 3)), as the store's
        // tensor map expects
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const uint32_t rbase = out_s + (h * NCH + c) * (BLOCK_M * 64) + row * 64;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int o = c * 32 + u * 8;
            const uint32_t addr = rbase + ((u ^ ((row >> 1) & 3)) << 4);
            if (c_in) {   // D = C + A B^T: the addend, added in fp32 before the rounding
              const uint4 cv = ld_shared_v4(addr);
              const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[o + 2 * e] += __uint_as_float(cw[e] << 16);
                acc[o + 2 * e + 1] += __uint_as_float(cw[e] & 0xFFFF0000u);
              }
            }
            uint32_t w0 = pack_bf16x2(acc[o + 0], acc[o + 1]);
            uint32_t w1 = pack_bf16x2(acc[o + 2], acc[o + 3]);
            uint32_t w2 = pack_bf16x2(acc[o + 4], acc[o + 5]);
            uint32_t w3 = pack_bf16x2(acc[o + 6], acc[o + 7]);
            if (zero_row) w0 = w1 = w2 = w3 = 0u;
            st_shared_v4(addr, w0, w1, w2, w3);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 32 * NUM_PROMO_WARPS);
        if (MODE != kMasked || T.rows == BLOCK_M) {
          // the store clips at the tensor's bounds (M rows, N columns).  Chunk
          // cc is stored by warp cc % NUM_PROMO_WARPS: a thread that issues a
          // TMA store stalls for a few hundred cycles, and one thread issuing
          // all of them would hold every promotion warp at the next tile's
          // first barrier.
          if (lane == 0 && !*abort_flag && T.rows > 0) {
            for (int cc = pw; cc < BN / 32; cc += NUM_PROMO_WARPS)
              if (T.n0 + cc * 32 < p.N)
                tma_store_3d(&tmD, out_s + cc * (BLOCK_M * 64), T.n0 + cc * 32, T.m0, T.zd);
            bulk_commit_group();
          }
        } else if (!*abort_flag) {
          // masked form, last tile of a group: rows >= masked_m[g] keep what D held
          constexpr int UPR = BN / 8;  // 16-byte units per row
          for (int i = pt; i < T.rows * UPR; i += 32 * NUM_PROMO_WARPS) {
            const int r = i / UPR, cu = i - r * UPR;
            const int n = T.n0 + cu * 8;
            if (n < p.N) {
              const uint32_t src = out_s + (cu >> 2) * (BLOCK_M * 64) + r * 64 +
                                   (((cu & 3) ^ ((r >> 1) & 3)) << 4);
              const uint4 w = ld_shared_v4(src);
              if constexpr (kDebug) {
                if (T.z >= p.num_groups || T.m0 + r >= p.M || n + 8 > p.N) {
                  raise_status(p, ST_DEBUG_BOUNDS);
                  continue;
                }
              }
              *reinterpret_cast<uint4*>(
                  p.D + (static_cast<size_t>(T.z) * p.M + T.m0 + r) * p.N + n) = w;
            }
          }
        }
      } else {
        // ------------- epilogue: K split over the cluster, DSMEM reduction ---
        // Each CTA owns a slice of R = ceil(rows / S) tile rows.  A CTA stages
        // its fp32 partial rows in its (now idle) operand ring, 16-byte unit u
        // of row r at unit u ^ (r & 7) (conflict-free row-per-thread writes),
        // and tells every CTA of the cluster so (READY, S arrivals, released
        // at cluster scope after a CTA barrier over the staging writes).  An
        // owner then reads its slice's rows from every CTA's staged partial
        // (its own locally, the others' through distributed shared memory),
        // sums them in rank order and stores bf16.  No CTA leaves before the
        // cluster's final rendezvous, so the partials stay readable until
        // every owner is done.  (Pushing the slices with bulk copies into
        // receive areas first took 1-2.8 us for the copies alone on the decode
        // shapes.)
        const int R = (T.rows + S - 1) / S;
        const int own_r0 = static_cast<int>(crank) * R;
        const int own_rows = max(0, min(T.rows, own_r0 + R) - own_r0);
        constexpr int ROWB = BN * 4;                       // bytes of one fp32 row
        const uint32_t stage_s = out_s;                    // [rows <= AROWS][BN] own partial
        named_bar_sync(1, 32 * NUM_PROMO_WARPS);           // this CTA's ring is idle
        if (row < T.rows) {
#pragma unroll
          for (int c = 0; c < HALF / 4; ++c) {
            const int u = h * (HALF / 4) + c;
            st_shared_v4(stage_s + row * ROWB + ((u ^ (row & 7)) << 4), __float_as_uint(acc[4 * c]),
                         __float_as_uint(acc[4 * c + 1]), __float_as_uint(acc[4 * c + 2]),
                         __float_as_uint(acc[4 * c + 3]));
          }
        }
        named_bar_sync(1, 32 * NUM_PROMO_WARPS);
        if (pt == 0)
          for (int r = 0; r < S; ++r) mbar_arrive_remote_release(bar(L::READY), r);
        wait_bar<true>(bar(L::READY), 0, abort_flag, p);
        __syncwarp();
        constexpr int UPR = BN / 4;  // 16-byte units per row
        constexpr int NPT_S = 32 * NUM_PROMO_WARPS;
        // An owner's slice has at most ceil(AROWS / 2) rows (S >= 2); the
        // units of a slice go to the threads in turn, MAX_IT per thread in
        // registers (a larger slice, S = 1, finishes in the loop after).
        constexpr int MAX_IT = ((AROWS + 1) / 2 * UPR + NPT_S - 1) / NPT_S;
        const int n_units = own_rows * UPR;
        // this thread's unit i: row rr of the slice, 16-byte unit cu; its
        // offset in a staged partial (same in every CTA)
        auto unit_off = [&](int i) -> uint32_t {
          const int rr = i / UPR, cu = i - rr * UPR;
          const int grow = own_r0 + rr;  // row in the tile (its swizzle key)
          return static_cast<uint32_t>(grow * ROWB + ((cu ^ (grow & 7)) << 4));
        };
        // bf16 of sum (+ C) for unit i, stored to D
        auto store_unit = [&](int i, float4 sum) {
          const int rr = i / UPR, cu = i - rr * UPR;
          const int grow = own_r0 + rr;
          const int n = T.n0 + cu * 4;
          if (n >= p.N) return;
          if (p.C != nullptr) {
            const uint2 c = __ldg(reinterpret_cast<const uint2*>(
                p.C + static_cast<size_t>(T.m0 + grow) * p.N + n));
            sum.x += __uint_as_float(c.x << 16);
            sum.y += __uint_as_float(c.x & 0xFFFF0000u);
            sum.z += __uint_as_float(c.y << 16);
            sum.w += __uint_as_float(c.y & 0xFFFF0000u);
          }
          if constexpr (kDebug) {
            if (T.m0 + grow >= p.M) {
              raise_status(p, ST_DEBUG_BOUNDS);
              return;
            }
          }
          if (!*abort_flag) {
            uint2 w;
            w.x = pack_bf16x2(sum.x, sum.y);
            w.y = pack_bf16x2(sum.z, sum.w);
            *reinterpret_cast<uint2*>(p.D + static_cast<size_t>(T.m0 + grow) * p.N + n) = w;
          }
        };
        // The S partials are added in rank order (deterministic), rank by
        // rank over all of this thread's units, so that each rank's loads
        // (local, or from a peer through distributed shared memory) are in
        // flight together.
        const uint8_t* stage_g = smem + L::OUT_OFF;     // this CTA's staged partial
        float4 sum[MAX_IT];
        for (int r = 0; r < S; ++r) {
          const uint8_t* src =
              r == static_cast<int>(crank)
                  ? stage_g
                  : static_cast<const uint8_t*>(__cluster_map_shared_rank(
                        const_cast<uint8_t*>(stage_g), static_cast<unsigned>(r)));
#pragma unroll
          for (int it = 0; it < MAX_IT; ++it) {
            const int i = pt + it * NPT_S;
            if (i < n_units) {
              const float4 v = *reinterpret_cast<const float4*>(src + unit_off(i));
              if (r == 0) {
                sum[it] = v;
              } else {
                sum[it].x += v.x; sum[it].y += v.y; sum[it].z += v.z; sum[it].w += v.w;
              }
            }
          }
        }
#pragma unroll
        for (int it = 0; it < MAX_IT; ++it) {
          const int i = pt + it * NPT_S;
          if (i < n_units) store_unit(i, sum[it]);
        }
        for (int i = pt + MAX_IT * NPT_S; i < n_units; i += NPT_S) {
          float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int r = 0; r < S; ++r) {
            const uint8_t* src =
                r == static_cast<int>(crank)
                    ? stage_g
                    : static_cast<const uint8_t*>(__cluster_map_shared_rank(
                          const_cast<uint8_t*>(stage_g), static_cast<unsigned>(r)));
            const float4 v = *reinterpret_cast<const float4*>(src + unit_off(i));
            if (r == 0) {
              acc4 = v;
            } else {
              acc4.x += v.x; acc4.y += v.y; acc4.z += v.z; acc4.w += v.w;
            }
          }
          store_unit(i, acc4);
        }
      }
    }  // tile loop
    // the staging tile must outlive the last stores' reads of it; their
    // writes need no wait here (they are performed before the grid counts as
    // complete, which is what a dependent launch and the host wait for)
    if (lane == 0) bulk_wait_group_read0();
    cp_async_wait_all();   // (after an abort, scale copies may still be in flight)
    __syncwarp();
  }

  // ----------------------------------------------------------- teardown --
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    else tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
  // No CTA leaves while a peer may still copy into it or read from it; every
  // exchanged byte has landed by now, so the rendezvous needs no memory
  // ordering.  All of a cluster's CTAs leave together: letting each thread
  // arrive as soon as its own part was done (and the sum overlap the peers'
  // skew) made back-to-back launches of 5-CTA clusters take a second wave
  // (decode 64x7168x16384, split 5: 29.5 -> 43 us).
  if (SPLIT || PAIR) cluster_sync_relaxed();
}

}  // namespace dgk

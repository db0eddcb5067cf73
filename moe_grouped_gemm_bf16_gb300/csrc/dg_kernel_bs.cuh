// The block-scaled form of the FP8 GEMM kernel for packed UE8M0 scales: the
// tensor cores apply the scales themselves (tcgen05.mma kind::mxf8f6f4 with
// block scaling) and accumulate each output tile over all of its K groups in
// tensor memory, so no per-group promotion runs on the CUDA cores.
//
// What it computes is the GEMM of the fp32-scale kernel with power-of-two
// scales (DeepGEMM, es.news.hada.io/topic?id=19459, "Interfaz GEMM y
// restricciones de layout": the SM100 kernels take the scales as packed
// UE8M0, four per 32-bit integer):
//   D[m,n] = bf16( [C[m,n] +] sum_g (A_g . B_g^T)[m,n] * 2^(ea[m,g]-127) * 2^(eb[n/128,g]-127) )
// A power-of-two scale applied to every product of a K group before the
// fp32 sum is the same product as the group's dot product times that scale,
// so the per-group scaling and the sum over groups run inside the MMA.
//
// Roles (512 threads; one persistent CTA per SM or one CTA pair per two SMs):
//   warps 0, 2  TMA producers (lane 0 of each, the stages of its parity): A
//               tile [128 x 128], B tile [BN x 128] (pair: the CTA's half of
//               B) into an S-stage ring; warp 2 first does the masked /
//               K-grouped set-up (device prefix sums).
//   warp 1      allocates tensor memory; lane 0 is an MMA issuer.
//   warp 3      lane 0 is the second MMA issuer when ISS = 2.
//               An issuer waits, per packed word (four K groups), for the
//               word's scale factors in its tensor-memory slot, then per K
//               group issues four block-scaled MMAs (K = 32 each) over the
//               whole tile width, committing the stage back to the producers,
//               the slot back to the scale-factor warp after the word's last
//               group and, after the tile's last group, its accumulator to
//               the epilogue.  With two issuers each takes every other K group
//               of a tile into an accumulator of its own (the thread that
//               issues tcgen05.mma stalls until the pipe takes it, and one
//               thread's loop per K group outlasts the MMAs of a 224- or
//               256-wide tile); the epilogue adds the two.
//   warps 4-11  epilogue: tensor memory -> (+ C) -> bf16 -> swizzled staging
//               buffer -> TMA store (masked tail tiles: row-guarded stores).
//   warp 12     scale factors: reads the packed words of the tile's rows
//               and B blocks from global memory, lays them out in shared
//               memory as the tensor-memory copies expect, and (lane 0) copies
//               them into each issuer's slot with tcgen05.cp once the slot's
//               previous MMAs have completed, committing the copies to the
//               issuer's barrier (so an issuer waits on one barrier per word
//               and issues nothing but MMAs and commits).
//
// Where the MMA reads its scale factors (measured on GB300 with distinct
// codes in every tensor-memory cell): the scale of A's row m from lane m,
// column [sfa] + m / 32; the scale of B's row n (output column n) from lane
// 32 q + n % 32 of the lane quarter q that computes the output row, column
// [sfb] + n / 32; in each 32-bit cell the byte the descriptor's scale-factor
// id names.  So a slot holds, per lane m, the packed word of row m in 4
// columns (each column read by one lane quarter), and, per 32-column chunk k
// of the tile, the packed word of that chunk's 128-column B block in column
// 4 + k of every lane (the tile may start inside a block).  With four K
// groups per packed word, K group g reads byte g % 4.
//
// Tensor memory: NACC x ISS accumulators of BN columns, then BS_SFT
// scale-factor slots of 16 columns (A in 4, B's 32-column chunks in up to 8
// more), BS_SFT / ISS for each issuer.
#pragma once
#include "dg_kernel.cuh"

namespace dgk {

constexpr int BS_SFS = 3;       // shared-memory slots of prepared scale factors
constexpr int BS_SFT = 4;       // tensor-memory scale-factor slots
constexpr int BS_SF_COLS = 16;  // tensor-memory columns per slot
constexpr int BS_SFB_COPIES = 2;  // 32 x 16-byte copies of B cells per slot (8 chunks of 32)
constexpr int BS_THREADS = 512;

template <int BN, int STAGES, bool PAIR, int NACC, int ISS = 1>
struct BsLayout {
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;   // rows of B held by one CTA
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K;
  static constexpr int B_BYTES = B_ROWS * BLOCK_K;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  // bf16 staging: one [128 rows x 32 columns] buffer per half of the epilogue
  static constexpr int OUT_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int STG_BYTES = BLOCK_M * 64;
  static constexpr int OUT_BYTES = 2 * STG_BYTES;
  static constexpr int SFA_BYTES = BLOCK_M * 16;            // 128 rows x 16 bytes
  static constexpr int SFB_BYTES = 32 * 16;                 // 32 rows x 4 cells of 4 bytes
  static constexpr int SFS_BYTES = SFA_BYTES + BS_SFB_COPIES * SFB_BYTES;
  static constexpr int SFS_OFF = OUT_OFF + OUT_BYTES;
  static constexpr int BAR_OFF = SFS_OFF + BS_SFS * SFS_BYTES;
  static constexpr int FULL = 0, EMPTY = STAGES, SFS_FULL = 2 * STAGES,
                       SFS_EMPTY = SFS_FULL + BS_SFS, SFT_EMPTY = SFS_EMPTY + BS_SFS,
                       SFT_FULL = SFT_EMPTY + BS_SFT, T_FULL = SFT_FULL + BS_SFT,
                       T_EMPTY = T_FULL + NACC, MMA_DONE = T_EMPTY + NACC, SF_DONE = MMA_DONE + 1,
                       NUM_BARS = SF_DONE + 1;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;   // [0] TMEM base, [1] abort flag
  // checked build: fill counters of the operand ring's and the staging ring's slots
  static constexpr int DBG_OFF = MISC_OFF + 16;
  static constexpr int DBG_BYTES = kDebug ? ((STAGES + BS_SFS) * 4 + 15) / 16 * 16 : 0;
  static constexpr int DYN_OFF = DBG_OFF + DBG_BYTES;       // masked / K-grouped tables
  static_assert(B_OFF % 1024 == 0 && OUT_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(SFS_OFF % 16 == 0 && BAR_OFF % 8 == 0, "alignment");
  static constexpr int SF_COL0 = NACC * ISS * BN;            // first scale-factor column
  static constexpr int SFT_PER = BS_SFT / ISS;               // scale-factor slots per issuer
  static_assert(SF_COL0 + BS_SFT * BS_SF_COLS <= 512, "tensor memory holds 512 columns");
  static_assert(ISS == 1 || (ISS == 2 && NACC == 1), "two issuers: one tile in flight");
  static constexpr int TMEM_COLS = 512;
};

// Dynamic shared memory of a block-scaled launch (host side too).
template <int BN, int STAGES, bool PAIR, int NACC, int ISS = 1>
__host__ __device__ constexpr int bs_smem_bytes(int num_groups, int mode) {
  return 1024 + BsLayout<BN, STAGES, PAIR, NACC, ISS>::DYN_OFF +
         (mode == kMasked ? (2 * num_groups + 1) * 4 : mode == kKGrouped ? (num_groups + 1) * 4 : 0);
}

template <int BN, int STAGES, int MODE, bool PAIR = false, int NACC = 1, int LAYOUT = kNT,
          int ISS = 1>
__global__ void __launch_bounds__(BS_THREADS, 1)
fp8_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ CUtensorMap tmC, const Params p) {
  static_assert(PROMO_WG == 2, "the epilogue uses warps 4-11");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN: a multiple of 32 in [64, 256]");
  static_assert(!PAIR || ((BN == 128 || BN == 224 || BN == 256) && LAYOUT == kNT &&
                          (MODE == kDense || MODE == kMasked)),
                "the pair form: dense or masked nt, 128-, 224- or 256-wide tiles");
  static_assert(BN / 32 <= 4 * BS_SFB_COPIES, "B scale cells of one slot");
  static_assert(LAYOUT == kNT || (BN % 128 == 0 && (MODE == kDense || MODE == kKGrouped)),
                "MN-major operands: dense or K-grouped, 128-multiple tiles");
  static_assert(MODE != kKGrouped || LAYOUT == kTN, "the K-grouped form is tn");
  static_assert(LAYOUT == kNT || (LAYOUT & 2) == 0 || BN % 128 == 0, "MN-major B: whole atoms");
  constexpr bool A_MN = (LAYOUT & 1) != 0;
  constexpr bool B_MN = (LAYOUT & 2) != 0;
  using L = BsLayout<BN, STAGES, PAIR, NACC, ISS>;
  // the epilogue's two warps per lane quarter split the tile's 32-column
  // chunks: the first takes ceil(NCHT / 2) of them, the second the rest
  constexpr int NCHT = BN / 32;
  constexpr int NCH0 = (NCHT + 1) / 2;
  constexpr uint32_t MN_ATOM_BYTES = 128 * BLOCK_K;
  constexpr uint64_t A_KSTEP = A_MN ? (32 * 128) >> 4 : 32 >> 4;
  constexpr uint64_t B_KSTEP = B_MN ? (32 * 128) >> 4 : 32 >> 4;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8 * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile uint32_t* abort_flag = misc + 1;
  int* prefix = reinterpret_cast<int*>(smem + L::DYN_OFF);
  int* mcnt = prefix + p.num_groups + 1;
  volatile uint32_t* dbg_fill = reinterpret_cast<volatile uint32_t*>(smem + L::DBG_OFF);
  volatile uint32_t* dbg_sfs_fill = dbg_fill + STAGES;

  const uint32_t crank = PAIR ? cluster_ctarank() : 0;
  constexpr int CL = PAIR ? 2 : 1;
  const bool leader = crank == 0;
  const int cluster_id = blockIdx.x / CL;
  const int num_clusters = gridDim.x / CL;

  // ------------------------------------------------------------- set-up --
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(L::FULL + s), 1);
      mbar_init(bar(L::EMPTY + s), 1);
    }
    for (int k = 0; k < BS_SFS; ++k) {
      mbar_init(bar(L::SFS_FULL + k), PAIR ? 2 : 1);   // pair: both CTAs' preparations
      mbar_init(bar(L::SFS_EMPTY + k), 1);             // the slot's copies have read it
    }
    for (int t = 0; t < BS_SFT; ++t) {
      mbar_init(bar(L::SFT_EMPTY + t), 1);
      mbar_init(bar(L::SFT_FULL + t), 1);
    }
    mbar_init(bar(L::SF_DONE), 1);
    for (int b = 0; b < NACC; ++b) {
      mbar_init(bar(L::T_FULL + b), ISS);
      mbar_init(bar(L::T_EMPTY + b), PAIR ? 2 * NUM_PROMO_WARPS : NUM_PROMO_WARPS);
    }
    mbar_init(bar(L::MMA_DONE), ISS);
    misc[1] = 0;
    if constexpr (kDebug)
      for (int i = 0; i < STAGES + BS_SFS; ++i) dbg_fill[i] = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
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
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (MODE == kMasked && warp == 2) {
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
    // first K group of every group: prefix sum of ks[g] / 128, checked and clamped
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
  if (PAIR) {
    cluster_arrive_relaxed();
    cluster_wait();
  }
  const uint32_t tmem_base = misc[0];
  const int num_m_blocks = (MODE == kMasked) ? prefix[p.num_groups] : p.num_m_blocks;
  const int num_tiles = num_m_blocks * p.num_n_blocks * (MODE == kKGrouped ? p.num_groups : 1);
  // tensor-memory address of scale-factor slot t of issuer e (lane 0)
  auto sf_col = [&](int e, int t) -> uint32_t {
    return tmem_base + static_cast<uint32_t>(L::SF_COL0 + (e * L::SFT_PER + t) * BS_SF_COLS);
  };

  if (warp == 0 || warp == 2) {
    // ----------------------------------------------------- TMA producers --
    // Two threads (warps 0 and 2) share the loads: a thread that issues a TMA
    // load stalls for ~250 cycles, so one thread issuing the two loads of
    // every K group falls behind the MMA.  Each owns the stages of its
    // parity, so every stage's latest fill is its owner's (the drain below
    // relies on it).
    if (lane == 0 && !(p.debug_flags & DBG_SKIP_PRODUCER)) {
      const int me = warp == 2 ? 1 : 0;
      uint32_t issued_mask = 0, issued_par = 0;
      int s = 0;
      uint32_t ph = 0;
      for (int t = cluster_id; t < num_tiles; t += num_clusters) {
        const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
        if (T.skip) continue;
        for (int g = T.kbeg; g < T.kend; ++g) {
          if ((s & 1) != me) {   // the other producer's stage
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
            const uint32_t a_dst = sbase + L::A_OFF + s * L::A_BYTES;
            const uint32_t b_dst = sbase + L::B_OFF + s * L::B_BYTES;
            if constexpr (PAIR) {
              // both CTAs' loads complete on the leader's FULL barrier; each
              // CTA holds half of the tile's B rows (the MMA's N: the
              // leader's half first)
              const uint32_t full = map_cluster(bar(L::FULL + s), 0);
              if (leader) mbar_arrive_expect_tx(bar(L::FULL + s), 2 * (L::A_BYTES + L::B_BYTES));
              tma_load_3d_pair(map_cluster(a_dst, crank), &tmA, full, g * BLOCK_K, T.m0, T.z);
              tma_load_3d_pair(map_cluster(b_dst, crank), &tmB, full, g * BLOCK_K,
                               T.n0 + static_cast<int>(crank) * (BN / 2), T.e);
            } else if constexpr (LAYOUT != kNT) {
              int nbox = 0;
              for (int bj = 0; bj < BN / 128; ++bj) nbox += (T.n0 + bj * 128 < p.N) ? 1 : 0;
              const uint32_t b_bytes = B_MN ? nbox * MN_ATOM_BYTES : L::B_BYTES;
              mbar_arrive_expect_tx(bar(L::FULL + s), L::A_BYTES + b_bytes);
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
              tma_load_3d(a_dst, &tmA, bar(L::FULL + s), g * BLOCK_K, T.m0, T.z);
              tma_load_3d(b_dst, &tmB, bar(L::FULL + s), g * BLOCK_K, T.n0, T.e);
            }
            issued_mask |= 1u << s;
            issued_par = (issued_par & ~(1u << s)) | (ph << s);
          }
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
      }
      for (int q = 0; q < STAGES; ++q)
        if (((issued_mask >> q) & 1u) && (!PAIR || leader))
          drain_wait(bar(L::FULL + q), (issued_par >> q) & 1u, p);
    }
    __syncwarp();
  } else if (warp == 1 || (ISS == 2 && warp == 3)) {
    // ------------------------------------------------------ MMA issuers ---
    // The issuing thread stalls on every tcgen05.mma until the tensor pipe
    // takes it, so the instructions between one K group's MMAs and the next
    // group's leave the pipe idle: the loop keeps them few (descriptors and
    // instruction descriptors precomputed, scale-factor work only at packed-
    // word boundaries, no per-group reads of the abort flag), and with
    // ISS = 2 two issuers take the K groups of a tile in turn.
    if (lane == 0 && (!PAIR || leader)) {
      const int e = warp == 3 ? 1 : 0;   // this issuer; its groups: (g - kbeg) % ISS == e
      int s = 0, b = 0;
      uint32_t ph = 0, bph = 0;
      uint32_t u = 0;           // scale-factor uses (packed words) so far
      uint32_t q = 0;           // K groups so far (checked build)
      const uint64_t ad0 = A_MN ? smem_desc_sw128_mnmajor(sbase + L::A_OFF, MN_ATOM_BYTES)
                                : smem_desc_sw128_kmajor(sbase + L::A_OFF);
      const uint64_t bd0 = B_MN ? smem_desc_sw128_mnmajor(sbase + L::B_OFF, MN_ATOM_BYTES)
                                : smem_desc_sw128_kmajor(sbase + L::B_OFF);
      for (int t = cluster_id; t < num_tiles; t += num_clusters) {
        const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
        if (T.skip) continue;
        const bool ok_t = wait_bar(bar(L::T_EMPTY + b), bph ^ 1, abort_flag, p);
        tc_fence_after();
        // the MMA's width: the tile, or its columns before N rounded up to 16
        // (the pair form splits B between the CTAs by the full width)
        const int nw = PAIR ? BN : min(BN, (p.N - T.n0 + 15) & ~15);
        const uint32_t idesc0 = idesc_mxf8f6f4(PAIR ? 2 * BLOCK_M : BLOCK_M, nw, A_MN, B_MN, 0, 0);
        const uint32_t d0 = tmem_base + static_cast<uint32_t>((b * ISS + e) * BN);
        int tt = 0;
        uint32_t sfa = 0;
        uint32_t acc = 0;         // this accumulator's first MMA of the tile starts it
        for (int g = T.kbeg; g < T.kend; ++g, ++q) {
          const bool mine = ISS == 1 || ((g - T.kbeg) & 1) == e;
          if (g == T.kbeg || (g & 3) == 0) {
            // a new packed word: the scale-factor warp has copied its scale
            // factors into this issuer's tensor-memory slot
            tt = static_cast<int>(u % L::SFT_PER);
            sfa = sf_col(e, tt);
            const bool ok_s = wait_bar(bar(L::SFT_FULL + e * L::SFT_PER + tt),
                                       (u / L::SFT_PER) & 1u, abort_flag, p);
            tc_fence_after();
            if constexpr (kDebug) {
              // the word's staging has been filled (at least) u / BS_SFS + 1 times
              if (ok_s && dbg_sfs_fill[u % BS_SFS] < u / BS_SFS + 1)
                dbg_fail(p, ST_DEBUG_PHASE, abort_flag);
            }
          }
          if (mine) {
            bool ok_f = wait_bar(bar(L::FULL + s), ph, abort_flag, p);
            tc_fence_after();
            if constexpr (kDebug) {
              if (ok_f && dbg_fill[s] != q / STAGES + 1) {
                dbg_fail(p, ST_DEBUG_PHASE, abort_flag);
                ok_f = false;
              }
            }
            if (ok_t && ok_f) {
              // descriptors of stage s: the start address field advances by
              // the stage offsets (>> 4); the group's byte of the packed word
              // picks both scales
              const uint64_t ad = ad0 + static_cast<uint64_t>((s * L::A_BYTES) >> 4);
              const uint64_t bd = bd0 + static_cast<uint64_t>((s * L::B_BYTES) >> 4);
              const uint32_t sfid = static_cast<uint32_t>(g & 3);
              const uint32_t idesc = idesc0 | (sfid << 4) | (sfid << 29);
#pragma unroll
              for (int kk = 0; kk < BLOCK_K / 32; ++kk) {
                if constexpr (PAIR)
                  mma_mxf8f6f4_bs_pair(d0, ad + A_KSTEP * kk, bd + B_KSTEP * kk, idesc, sfa,
                                       sfa + 4, acc | kk);
                else
                  mma_mxf8f6f4_bs(d0, ad + A_KSTEP * kk, bd + B_KSTEP * kk, idesc, sfa, sfa + 4,
                                  acc | kk);
              }
              acc = 1;
            }
            if constexpr (PAIR) mma_commit_pair_multicast(bar(L::EMPTY + s), 0x3);
            else mma_commit(bar(L::EMPTY + s));
          }
          if (g == T.kend - 1 || (g & 3) == 3) {
            // the word's last group: its tensor-memory slot frees up once these MMAs complete
            if constexpr (PAIR) mma_commit_pair_multicast(bar(L::SFT_EMPTY + e * L::SFT_PER + tt), 0x1);
            else mma_commit(bar(L::SFT_EMPTY + e * L::SFT_PER + tt));
            ++u;
          }
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
        // the tile's accumulator to the epilogue (pair: in both CTAs)
        if constexpr (PAIR) mma_commit_pair_multicast(bar(L::T_FULL + b), 0x3);
        else mma_commit(bar(L::T_FULL + b));
        if (++b == NACC) { b = 0; bph ^= 1; }
      }
      if constexpr (PAIR) mma_commit_pair_multicast(bar(L::MMA_DONE), 0x1);
      else mma_commit(bar(L::MMA_DONE));
      drain_wait(bar(L::MMA_DONE), 0, p);
    }
    __syncwarp();
  } else if (warp == 12) {
    // -------------------------------------------- scale-factor preparation --
    // Per packed word of a tile: the A scale word of each of the tile's 128
    // rows into the four 32-bit cells of its 16-byte row (copied to lane m,
    // columns 0-3, by tcgen05.cp 128x128b), and for the tile's 32-column
    // chunk k the word of its B block into cell k % 4 of every row of copy
    // k / 4 (copied to every lane quarter, column 4 + k, by 32x128b.warpx4).
    // Lane 0 then issues those copies itself, into the tensor-memory slot of
    // each issuer with a K group in the word, once the slot's previous MMAs
    // have completed, and commits them to the issuers' barriers: the issuer
    // only waits for one barrier per word (its thread stalls on every
    // instruction between its MMAs).  Pair form: the leader's lane 0 copies
    // both CTAs' staging (cta_group::2) once both are filled.
    const uint32_t* sfa = reinterpret_cast<const uint32_t*>(p.sa_packed);
    const uint32_t* sfb = reinterpret_cast<const uint32_t*>(p.sb);
    uint32_t u = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters) {
      const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
      if (T.skip) continue;
      for (int w0 = T.kbeg >> 2; w0 <= (T.kend - 1) >> 2; ++w0, ++u) {
        const int k = static_cast<int>(u % BS_SFS);
        wait_bar(bar(L::SFS_EMPTY + k), ((u / BS_SFS) & 1u) ^ 1u, abort_flag, p);
        const uint32_t dst = sbase + L::SFS_OFF + k * L::SFS_BYTES;
        uint32_t wa[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int m = T.m0 + lane + 32 * r;
          wa[r] = m < p.M ? __ldg(sfa + (static_cast<size_t>(T.z) * p.kbp + w0) * p.ld_sa + m)
                          : 0x7F7F7F7Fu;   // rows past M: scale 1 (never stored)
        }
        uint32_t wb = 0;
        if (lane < BN / 32) {
          // the B block of the tile's 32-column chunk `lane` (chunks past N
          // take the last block: their columns are never stored)
          const int blk = min((T.n0 + 32 * lane) >> 7, p.nb - 1);
          wb = __ldg(sfb + (static_cast<size_t>(T.e) * p.nb + blk) * p.kbp + w0);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) st_shared_v4(dst + (lane + 32 * r) * 16, wa[r], wa[r], wa[r], wa[r]);
#pragma unroll
        for (int j = 0; j < (BN / 32 + 3) / 4; ++j) {
          const uint32_t c0 = __shfl_sync(0xffffffffu, wb, 4 * j);
          const uint32_t c1 = __shfl_sync(0xffffffffu, wb, 4 * j + 1);
          const uint32_t c2 = __shfl_sync(0xffffffffu, wb, 4 * j + 2);
          const uint32_t c3 = __shfl_sync(0xffffffffu, wb, 4 * j + 3);
          st_shared_v4(dst + L::SFA_BYTES + j * L::SFB_BYTES + lane * 16, c0, c1, c2, c3);
        }
        fence_proxy_async_smem();   // the copies read through the async proxy
        __syncwarp();
        if constexpr (kDebug) {
          if (lane == 0) dbg_sfs_fill[k] = dbg_sfs_fill[k] + 1;
        }
        if (lane == 0) {
          if (PAIR && !leader) {
            mbar_arrive_remote_release(bar(L::SFS_FULL + k), 0);
          } else {
            bool ok = true;
            if constexpr (PAIR) {
              mbar_arrive(bar(L::SFS_FULL + k));
              ok = wait_bar<true>(bar(L::SFS_FULL + k), (u / BS_SFS) & 1u, abort_flag, p);
            }
            const int tt = static_cast<int>(u % L::SFT_PER);
            // the issuers with a K group in this word (two issuers: by parity)
            const int g0 = max(T.kbeg, w0 * 4), g1 = min(T.kend, w0 * 4 + 4);
            for (int e = 0; e < ISS; ++e) {
              const bool has = ISS == 1 || g1 - g0 >= 2 || ((g0 - T.kbeg) & 1) == e;
              if (u >= L::SFT_PER)   // the slot's previous MMAs have completed
                ok = wait_bar(bar(L::SFT_EMPTY + e * L::SFT_PER + tt), ((u / L::SFT_PER) - 1) & 1u,
                              abort_flag, p) && ok;
              tc_fence_after();
              if (has && ok) {
                const uint32_t tsf = sf_col(e, tt);
                if constexpr (PAIR) {
                  tmem_cp_128x128b_pair(tsf, smem_desc_rows16(dst, 128));
#pragma unroll
                  for (int j = 0; j < (BN / 32 + 3) / 4; ++j)
                    tmem_cp_32x128b_warpx4_pair(
                        tsf + 4 + 4 * j, smem_desc_rows16(dst + L::SFA_BYTES + j * L::SFB_BYTES, 128));
                } else {
                  tmem_cp_128x128b(tsf, smem_desc_rows16(dst, 128));
#pragma unroll
                  for (int j = 0; j < (BN / 32 + 3) / 4; ++j)
                    tmem_cp_32x128b_warpx4(
                        tsf + 4 + 4 * j, smem_desc_rows16(dst + L::SFA_BYTES + j * L::SFB_BYTES, 128));
                }
              }
              // (every word completes a phase of every issuer's slot barrier)
              if constexpr (PAIR) mma_commit_pair_multicast(bar(L::SFT_FULL + e * L::SFT_PER + tt), 0x1);
              else mma_commit(bar(L::SFT_FULL + e * L::SFT_PER + tt));
            }
            // the staging slot is free once the copies have read it (pair: in both CTAs)
            if constexpr (PAIR) mma_commit_pair_multicast(bar(L::SFS_EMPTY + k), 0x3);
            else mma_commit(bar(L::SFS_EMPTY + k));
          }
        }
      }
    }
    if (lane == 0 && (!PAIR || leader)) {
      // the last copies have completed before the tensor memory is freed
      if constexpr (PAIR) mma_commit_pair_multicast(bar(L::SF_DONE), 0x1);
      else mma_commit(bar(L::SF_DONE));
      drain_wait(bar(L::SF_DONE), 0, p);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------- epilogue ---
    // Two warps per lane quarter: warps 4-7 (half 0) and 8-11 (half 1) each
    // cover all 128 rows (thread = row) of their share of the tile's 32-column
    // chunks.  Per tile: this thread's row of the addend C for its chunks is
    // prefetched into registers while the MMAs run; the accumulator's chunks
    // are read from tensor memory, (+ C) rounded to bf16 into registers, and
    // the accumulator handed back at once; then each chunk goes out through
    // the half's [128 x 32] staging buffer (64-byte swizzle) and a TMA store
    // (masked tail tiles: row-guarded 16-byte stores straight from registers).
    const int q = warp & 3;             // TMEM lane quadrant this warp may access
    const int h = (warp - 4) >> 2;      // which share of the tile's column chunks
    const int c_lo = h ? NCH0 : 0;
    const int nch = h ? NCHT - NCH0 : NCH0;
    const int row = q * 32 + lane;
    const bool hlead = q == 0 && lane == 0;   // issues the half's TMA stores
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t stg = sbase + L::OUT_OFF + h * L::STG_BYTES;
    int b = 0;
    uint32_t bph = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters) {
      const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
      const bool has_c = (MODE == kDense || MODE == kKGrouped) && p.C != nullptr;
      const int m = T.m0 + row;
      uint32_t pk[NCH0][16];   // this thread's chunks as bf16 pairs (first the addend)
#pragma unroll
      for (int i = 0; i < NCH0; ++i) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int n = T.n0 + (c_lo + i) * 32 + u * 8;
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (has_c && i < nch && m < p.M && n < p.N)
            w = __ldg(reinterpret_cast<const uint4*>(
                p.C + (static_cast<size_t>(T.zd) * p.M + m) * p.N + n));
          pk[i][4 * u] = w.x;
          pk[i][4 * u + 1] = w.y;
          pk[i][4 * u + 2] = w.z;
          pk[i][4 * u + 3] = w.w;
        }
      }
      // contiguous: padding blocks and rows (m_indices = -1) and bad experts are +0
      bool zero_row = MODE == kContiguous && T.skip != 0;
      if constexpr (MODE == kContiguous) {
        if (T.skip == 2 && h == 0 && row == 0) raise_status(p, ST_EXPERT_RANGE);
        if (!T.skip) {
          const int id = __ldg(p.m_indices + m);
          if (id != T.e) {
            zero_row = true;
            if (id >= 0) raise_status(p, ST_EXPERT_RANGE);
          }
        }
      }
      const bool acc_in = !T.skip && wait_bar(bar(L::T_FULL + b), bph, abort_flag, p);
      // with two issuers the second accumulator holds the tile's odd K groups
      const bool two = ISS == 2 && T.kend - T.kbeg >= 2;
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < NCH0; ++i) {
        if (ISS == 1 && i < nch) {
          // one accumulator: the whole 32-column chunk per load (each wait
          // for a tensor-memory load exposes its latency, and the next tile's
          // MMAs wait for the last of them)
          uint32_t v[32];
          if (acc_in) {
            tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(b * BN + (c_lo + i) * 32), v);
            tmem_wait_ld(v);
          } else {
#pragma unroll
            for (int e2 = 0; e2 < 32; ++e2) v[e2] = 0u;
          }
          if (i == nch - 1 && !T.skip) {
            // every tensor-memory load of this warp has completed: hand the
            // accumulator back (pair: on the leader's barrier)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (PAIR && !leader) mbar_arrive_remote_relaxed(bar(L::T_EMPTY + b), 0);
              else mbar_arrive(bar(L::T_EMPTY + b));
            }
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            // D = C + A B: the addend added in fp32, then one rounding
            const uint32_t cw = pk[i][e];
            const float lo = __uint_as_float(v[2 * e]) + __uint_as_float(cw << 16);
            const float hi = __uint_as_float(v[2 * e + 1]) + __uint_as_float(cw & 0xFFFF0000u);
            pk[i][e] = zero_row ? 0u : pack_bf16x2(lo, hi);
          }
        } else if (i < nch) {
          // two accumulators: the chunk in two 16-column halves (registers:
          // the second accumulator's half rides along)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[16];
            if (acc_in) {
              const uint32_t col =
                  t_lane + static_cast<uint32_t>(b * ISS * BN + (c_lo + i) * 32 + 16 * hh);
              tmem_ld_32x32b_x16(col, v);
              if constexpr (ISS == 2) {
                uint32_t w[16];
                if (two) tmem_ld_32x32b_x16(col + BN, w);
                tmem_wait_ld16(v);
                if (two) {
                  tmem_wait_ld16(w);
#pragma unroll
                  for (int e2 = 0; e2 < 16; ++e2)
                    v[e2] = __float_as_uint(__uint_as_float(v[e2]) + __uint_as_float(w[e2]));
                }
              } else {
                tmem_wait_ld16(v);
              }
            } else {
#pragma unroll
              for (int e2 = 0; e2 < 16; ++e2) v[e2] = 0u;
            }
            if (i == nch - 1 && hh == 1 && !T.skip) {
              // every tensor-memory load of this warp has completed: hand the
              // accumulator back (pair: on the leader's barrier)
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                if (PAIR && !leader) mbar_arrive_remote_relaxed(bar(L::T_EMPTY + b), 0);
                else mbar_arrive(bar(L::T_EMPTY + b));
              }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              // D = C + A B: the addend added in fp32, then one rounding
              const uint32_t cw = pk[i][8 * hh + e];
              const float lo = __uint_as_float(v[2 * e]) + __uint_as_float(cw << 16);
              const float hi = __uint_as_float(v[2 * e + 1]) + __uint_as_float(cw & 0xFFFF0000u);
              pk[i][8 * hh + e] = zero_row ? 0u : pack_bf16x2(lo, hi);
            }
          }
        }
      }
      if (!T.skip) {
        if (++b == NACC) { b = 0; bph ^= 1; }
      }
      if (MODE == kMasked && T.rows < BLOCK_M) {
        // masked form, last tile of a group: rows >= masked_m[g] keep what D held
        if (row < T.rows && !*abort_flag) {
#pragma unroll
          for (int i = 0; i < NCH0; ++i) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int n = T.n0 + (c_lo + i) * 32 + u * 8;
              if (i < nch && n < p.N) {
                if constexpr (kDebug) {
                  if (T.z >= p.num_groups || m >= p.M || n + 8 > p.N) {
                    raise_status(p, ST_DEBUG_BOUNDS);
                    continue;
                  }
                }
                *reinterpret_cast<uint4*>(p.D + (static_cast<size_t>(T.z) * p.M + m) * p.N + n) =
                    make_uint4(pk[i][4 * u], pk[i][4 * u + 1], pk[i][4 * u + 2], pk[i][4 * u + 3]);
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < NCH0; ++i) {
          if (i < nch && T.n0 + (c_lo + i) * 32 < p.N && T.rows > 0) {
            // the staging buffer is free once the half's previous store has read it
            if (hlead) bulk_wait_group_read0();
            named_bar_sync(2 + h, 128);
            // [128 rows x 64 B], 16-byte unit u of row r at unit u ^ ((r >> 1) & 3)
            const uint32_t rbase = stg + row * 64;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              st_shared_v4(rbase + ((u ^ ((row >> 1) & 3)) << 4), pk[i][4 * u], pk[i][4 * u + 1],
                           pk[i][4 * u + 2], pk[i][4 * u + 3]);
            fence_proxy_async_smem();
            named_bar_sync(2 + h, 128);
            if (hlead && !*abort_flag) {
              tma_store_3d(&tmD, stg, T.n0 + (c_lo + i) * 32, T.m0, T.zd);
              bulk_commit_group();
            }
          }
        }
      }
    }
    // (the staging must outlive the last stores' reads; their writes are
    // performed before the grid counts as complete)
    if (hlead) bulk_wait_group_read0();
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
  if (PAIR) cluster_sync_relaxed();
}

}  // namespace dgk

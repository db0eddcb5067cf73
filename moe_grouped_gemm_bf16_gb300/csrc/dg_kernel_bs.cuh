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
// Roles (384 threads; one persistent CTA per SM or one CTA pair per two SMs):
//   warp 0      TMA producer: A tile [128 x 128], B tile [BN x 128] (pair: the
//               CTA's half of B, in 64-row boxes) into an S-stage ring.
//   warp 1      allocates tensor memory; lane 0 issues, per group of four K
//               groups (one packed scale word), the copies of the prepared
//               scale factors into tensor memory, then per K group the
//               block-scaled MMAs (one per 128-column block of B the tile
//               touches, each with one B scale), committing the stage back to
//               the producer and, after the tile's last group, the
//               accumulator to the epilogue.
//   warp 2      masked / K-grouped set-up (device prefix sums), then idle.
//   warp 3      scale-factor preparation: reads the packed words of the
//               tile's rows and B blocks from global memory and lays them out
//               in shared memory as the tensor-memory copies expect, every
//               word in each of a row's four cells (so the layout holds
//               whichever tensor-memory column a lane quarter reads).
//   warps 4-11  epilogue: tensor memory -> (+ C) -> bf16 -> swizzled staging
//               tile -> TMA store (masked tail tiles: row-guarded stores).
//
// Tensor memory: NACC accumulators of BN columns, then BS_SFT scale-factor
// slots of 16 columns (the A scales in 4 columns, each B block's in 4 more).
#pragma once
#include "dg_kernel.cuh"

namespace dgk {

constexpr int BS_SFS = 3;       // shared-memory slots of prepared scale factors
constexpr int BS_SFT = 4;       // tensor-memory scale-factor slots
constexpr int BS_SF_COLS = 16;  // tensor-memory columns per slot
constexpr int BS_MAX_BLK = 3;   // 128-column B blocks a tile may touch

template <int BN, int STAGES, bool PAIR, int NACC>
struct BsLayout {
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;   // rows of B held by one CTA
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K;
  static constexpr int B_BYTES = B_ROWS * BLOCK_K;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int OUT_OFF = B_OFF + STAGES * B_BYTES;   // bf16 staging, [BN/32][128][64 B]
  static constexpr int OUT_BYTES = BLOCK_M * BN * 2;
  static constexpr int SFA_BYTES = BLOCK_M * 16;            // 128 rows x 16 bytes
  static constexpr int SFB_BYTES = 32 * 16;                 // 32 rows x 16 bytes per B block
  static constexpr int SFS_BYTES = SFA_BYTES + BS_MAX_BLK * SFB_BYTES;
  static constexpr int SFS_OFF = OUT_OFF + OUT_BYTES;
  static constexpr int BAR_OFF = SFS_OFF + BS_SFS * SFS_BYTES;
  static constexpr int FULL = 0, EMPTY = STAGES, SFS_FULL = 2 * STAGES,
                       SFS_EMPTY = SFS_FULL + BS_SFS, SFT_EMPTY = SFS_EMPTY + BS_SFS,
                       T_FULL = SFT_EMPTY + BS_SFT, T_EMPTY = T_FULL + NACC,
                       MMA_DONE = T_EMPTY + NACC, C_FULL = MMA_DONE + 1, NUM_BARS = C_FULL + 1;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;   // [0] TMEM base, [1] abort flag
  // checked build: fill counters of the operand ring's and the staging ring's slots
  static constexpr int DBG_OFF = MISC_OFF + 16;
  static constexpr int DBG_BYTES = kDebug ? ((STAGES + BS_SFS) * 4 + 15) / 16 * 16 : 0;
  static constexpr int DYN_OFF = DBG_OFF + DBG_BYTES;       // masked / K-grouped tables
  static_assert(B_OFF % 1024 == 0 && OUT_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(SFS_OFF % 16 == 0 && BAR_OFF % 8 == 0, "alignment");
  static constexpr int SF_COL0 = NACC * BN;                  // first scale-factor column
  static_assert(SF_COL0 + BS_SFT * BS_SF_COLS <= 512, "tensor memory holds 512 columns");
  static constexpr int TMEM_COLS = 512;
};

// Dynamic shared memory of a block-scaled launch (host side too).
template <int BN, int STAGES, bool PAIR, int NACC>
__host__ __device__ constexpr int bs_smem_bytes(int num_groups, int mode) {
  return 1024 + BsLayout<BN, STAGES, PAIR, NACC>::DYN_OFF +
         (mode == kMasked ? (2 * num_groups + 1) * 4 : mode == kKGrouped ? (num_groups + 1) * 4 : 0);
}

// The 128-column B blocks a tile [n0, n0 + BN) touches, as column ranges of
// the tile: sub-MMA j covers tile columns [c0[j], c0[j] + w[j]), all in block
// (n0 + c0[j]) / 128, and only those that start before N.
struct SubMmas {
  int n;
  int c0[BS_MAX_BLK];
  int w[BS_MAX_BLK];
};

template <int BN>
__device__ __forceinline__ SubMmas sub_mmas(int n0, int N) {
  SubMmas s;
  s.n = 0;
  int c = 0;
#pragma unroll
  for (int j = 0; j < BS_MAX_BLK; ++j) {
    if (c < BN && n0 + c < N) {
      const int w = min(BN - c, 128 - ((n0 + c) & 127));
      s.c0[s.n] = c;
      s.w[s.n] = w;
      ++s.n;
      c += w;
    }
  }
  return s;
}

template <int BN, int STAGES, int MODE, bool PAIR = false, int NACC = 1, int LAYOUT = kNT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
fp8_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ CUtensorMap tmC, const Params p) {
  static_assert(PROMO_WG == 2, "the epilogue uses warps 4-11");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN: a multiple of 32 in [64, 256]");
  static_assert(!PAIR || ((BN == 128 || BN == 256) && LAYOUT == kNT &&
                          (MODE == kDense || MODE == kMasked)),
                "the pair form: dense or masked nt, 128- or 256-wide tiles");
  static_assert(LAYOUT == kNT || (BN % 128 == 0 && (MODE == kDense || MODE == kKGrouped)),
                "MN-major operands: dense or K-grouped, 128-multiple tiles");
  static_assert(MODE != kKGrouped || LAYOUT == kTN, "the K-grouped form is tn");
  static_assert(LAYOUT == kNT || (LAYOUT & 2) == 0 || BN % 128 == 0, "MN-major B: whole atoms");
  constexpr bool A_MN = (LAYOUT & 1) != 0;
  constexpr bool B_MN = (LAYOUT & 2) != 0;
  using L = BsLayout<BN, STAGES, PAIR, NACC>;
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
      mbar_init(bar(L::SFS_EMPTY + k), 1);
    }
    for (int t = 0; t < BS_SFT; ++t) mbar_init(bar(L::SFT_EMPTY + t), 1);
    for (int b = 0; b < NACC; ++b) {
      mbar_init(bar(L::T_FULL + b), 1);
      mbar_init(bar(L::T_EMPTY + b), PAIR ? 2 * NUM_PROMO_WARPS : NUM_PROMO_WARPS);
    }
    mbar_init(bar(L::MMA_DONE), 1);
    mbar_init(bar(L::C_FULL), 1);
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
  // tensor-memory address of scale-factor slot t (lane 0)
  auto sf_col = [&](int t) -> uint32_t {
    return tmem_base + static_cast<uint32_t>(L::SF_COL0 + t * BS_SF_COLS);
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && !(p.debug_flags & DBG_SKIP_PRODUCER)) {
      uint32_t issued_mask = 0, issued_par = 0;
      int s = 0;
      uint32_t ph = 0;
      for (int t = cluster_id; t < num_tiles; t += num_clusters) {
        const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
        if (T.skip) continue;
        for (int g = T.kbeg; g < T.kend; ++g) {
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
              // both CTAs' loads complete on the leader's FULL barrier; this
              // CTA's B rows: in each 128-column block j of the tile, the
              // 64-row half `crank` (so each pair MMA reads one block)
              const uint32_t full = map_cluster(bar(L::FULL + s), 0);
              if (leader) mbar_arrive_expect_tx(bar(L::FULL + s), 2 * (L::A_BYTES + L::B_BYTES));
              tma_load_3d_pair(map_cluster(a_dst, crank), &tmA, full, g * BLOCK_K, T.m0, T.z);
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tma_load_3d_pair(map_cluster(b_dst + j * 64 * BLOCK_K, crank), &tmB, full,
                                 g * BLOCK_K, T.n0 + j * 128 + static_cast<int>(crank) * 64, T.e);
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
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ---
    if (lane == 0 && (!PAIR || leader)) {
      int s = 0, b = 0;
      uint32_t ph = 0, bph = 0;
      uint32_t u = 0;           // scale-factor uses (packed words) so far
      uint32_t q = 0;           // K groups so far (checked build)
      for (int t = cluster_id; t < num_tiles; t += num_clusters) {
        const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
        if (T.skip) continue;
        const bool ok_t = wait_bar(bar(L::T_EMPTY + b), bph ^ 1, abort_flag, p);
        tc_fence_after();
        const SubMmas sm = sub_mmas<BN>(T.n0, p.N);
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(b * BN);
        int k = 0, tt = 0;
        for (int g = T.kbeg; g < T.kend; ++g) {
          if (g == T.kbeg || (g & 3) == 0) {
            // a new packed word: its prepared scale factors into tensor memory
            k = static_cast<int>(u % BS_SFS);
            tt = static_cast<int>(u % BS_SFT);
            if (u >= BS_SFT)   // the slot's previous MMAs have completed
              wait_bar(bar(L::SFT_EMPTY + tt), ((u / BS_SFT) - 1) & 1u, abort_flag, p);
            bool ok_s = PAIR ? wait_bar<true>(bar(L::SFS_FULL + k), (u / BS_SFS) & 1u,
                                              abort_flag, p)
                             : wait_bar(bar(L::SFS_FULL + k), (u / BS_SFS) & 1u, abort_flag, p);
            tc_fence_after();
            if constexpr (kDebug) {
              if (ok_s && dbg_sfs_fill[k] != u / BS_SFS + 1) {
                dbg_fail(p, ST_DEBUG_PHASE, abort_flag);
                ok_s = false;
              }
            }
            if (ok_s && ok_t) {
              const uint32_t src = sbase + L::SFS_OFF + k * L::SFS_BYTES;
              if constexpr (PAIR) {
                tmem_cp_128x128b_pair(sf_col(tt), smem_desc_rows16(src, 128));
#pragma unroll
                for (int j = 0; j < BS_MAX_BLK; ++j)
                  if (j < sm.n)
                    tmem_cp_32x128b_warpx4_pair(
                        sf_col(tt) + 4 + 4 * j,
                        smem_desc_rows16(src + L::SFA_BYTES + j * L::SFB_BYTES, 128));
              } else {
                tmem_cp_128x128b(sf_col(tt), smem_desc_rows16(src, 128));
#pragma unroll
                for (int j = 0; j < BS_MAX_BLK; ++j)
                  if (j < sm.n)
                    tmem_cp_32x128b_warpx4(
                        sf_col(tt) + 4 + 4 * j,
                        smem_desc_rows16(src + L::SFA_BYTES + j * L::SFB_BYTES, 128));
              }
            }
          }
          bool ok_f = wait_bar(bar(L::FULL + s), ph, abort_flag, p);
          tc_fence_after();
          if constexpr (kDebug) {
            if (ok_f && dbg_fill[s] != q / STAGES + 1) {
              dbg_fail(p, ST_DEBUG_PHASE, abort_flag);
              ok_f = false;
            }
          }
          ++q;
          if (ok_t && ok_f && !*abort_flag) {
            const uint32_t a_src = sbase + L::A_OFF + s * L::A_BYTES;
            const uint32_t b_src = sbase + L::B_OFF + s * L::B_BYTES;
            const uint64_t ad = A_MN ? smem_desc_sw128_mnmajor(a_src, MN_ATOM_BYTES)
                                     : smem_desc_sw128_kmajor(a_src);
            const uint32_t sfid = static_cast<uint32_t>(g & 3);   // the group's byte of the word
#pragma unroll
            for (int j = 0; j < BS_MAX_BLK; ++j) {
              if (j >= sm.n) break;
              // sub-MMA j: B rows of its block (pair: 64 per CTA), its own B scale
              uint32_t bsrc;
              if constexpr (PAIR) bsrc = b_src + j * 64 * BLOCK_K;
              else if constexpr (B_MN) bsrc = b_src + (sm.c0[j] >> 7) * MN_ATOM_BYTES;
              else bsrc = b_src + sm.c0[j] * BLOCK_K;
              const uint64_t bd = B_MN ? smem_desc_sw128_mnmajor(bsrc, MN_ATOM_BYTES)
                                       : smem_desc_sw128_kmajor(bsrc);
              const uint32_t idesc =
                  idesc_mxf8f6f4(PAIR ? 2 * BLOCK_M : BLOCK_M, sm.w[j], A_MN, B_MN, sfid, sfid);
              const uint32_t d = d0 + static_cast<uint32_t>(sm.c0[j]);
              const uint32_t sfb = sf_col(tt) + 4 + 4 * j;
#pragma unroll
              for (int kk = 0; kk < BLOCK_K / 32; ++kk) {
                const uint32_t acc = (g > T.kbeg || kk > 0) ? 1u : 0u;
                if constexpr (PAIR)
                  mma_mxf8f6f4_bs_pair(d, ad + A_KSTEP * kk, bd + B_KSTEP * kk, idesc, sf_col(tt),
                                       sfb, acc);
                else
                  mma_mxf8f6f4_bs(d, ad + A_KSTEP * kk, bd + B_KSTEP * kk, idesc, sf_col(tt), sfb,
                                  acc);
              }
            }
          }
          if constexpr (PAIR) mma_commit_pair_multicast(bar(L::EMPTY + s), 0x3);
          else mma_commit(bar(L::EMPTY + s));
          if (g == T.kend - 1 || (g & 3) == 3) {
            // the word's last group: its staging slot and tensor-memory slot free up
            if constexpr (PAIR) {
              mma_commit_pair_multicast(bar(L::SFS_EMPTY + k), 0x3);
              mma_commit_pair_multicast(bar(L::SFT_EMPTY + tt), 0x1);
            } else {
              mma_commit(bar(L::SFS_EMPTY + k));
              mma_commit(bar(L::SFT_EMPTY + tt));
            }
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
  } else if (warp == 3) {
    // -------------------------------------------- scale-factor preparation --
    // Per packed word of a tile: the A scale word of each of the tile's 128
    // rows into four 32-bit cells of its 16-byte row, and each B block's word
    // into every cell of its 32 x 16-byte block (then copied by the MMA
    // issuer with tcgen05.cp: 128x128b for A, 32x128b.warpx4 for B).
    const uint32_t* sfa = reinterpret_cast<const uint32_t*>(p.sa_packed);
    const uint32_t* sfb = reinterpret_cast<const uint32_t*>(p.sb);
    uint32_t u = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters) {
      const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
      if (T.skip) continue;
      const SubMmas sm = sub_mmas<BN>(T.n0, p.N);
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
        if (lane < sm.n) {
          // sub-MMA `lane`'s B block: the tile's first block plus the lane
          // (the sub-MMAs cover consecutive blocks)
          const int blk = min((T.n0 >> 7) + lane, p.nb - 1);
          wb = __ldg(sfb + (static_cast<size_t>(T.e) * p.nb + blk) * p.kbp + w0);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) st_shared_v4(dst + (lane + 32 * r) * 16, wa[r], wa[r], wa[r], wa[r]);
#pragma unroll
        for (int j = 0; j < BS_MAX_BLK; ++j) {
          const uint32_t w = __shfl_sync(0xffffffffu, wb, j);
          if (j < sm.n) st_shared_v4(dst + L::SFA_BYTES + j * L::SFB_BYTES + lane * 16, w, w, w, w);
        }
        fence_proxy_async_smem();   // the copies read through the async proxy
        __syncwarp();
        if constexpr (kDebug) {
          if (lane == 0) dbg_sfs_fill[k] = dbg_sfs_fill[k] + 1;
        }
        if (lane == 0) {
          if (PAIR && !leader) mbar_arrive_remote_release(bar(L::SFS_FULL + k), 0);
          else mbar_arrive(bar(L::SFS_FULL + k));
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------- epilogue ---
    const int q = warp & 3;             // TMEM lane quadrant this warp may access
    const int h = (warp - 4) >> 2;      // which share of the tile's column chunks
    const int c_lo = h ? NCH0 : 0, c_hi = h ? NCHT : NCH0;
    const int row = q * 32 + lane;
    const int ept = threadIdx.x - 128;  // 0 .. 255
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t out_s = sbase + L::OUT_OFF;
    int b = 0;
    uint32_t bph = 0, cph = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters) {
      const Tile T = decode_tile<BN, MODE, PAIR>(t, p, num_m_blocks, prefix, mcnt, 0, p.kb, crank);
      const bool has_c = (MODE == kDense || MODE == kKGrouped) && p.C != nullptr;
      // the previous tile's store has read the staging tile; the addend of
      // this tile (D = C + A B) goes into it, in the store's own layout
      if (ept == 0) {
        bulk_wait_group_read0();
        if (has_c) {
          uint32_t bytes = 0;
          for (int cc = 0; cc < BN / 32; ++cc)
            if (T.n0 + cc * 32 < p.N) bytes += BLOCK_M * 64;
          mbar_arrive_expect_tx(bar(L::C_FULL), bytes);
          for (int cc = 0; cc < BN / 32; ++cc)
            if (T.n0 + cc * 32 < p.N)
              tma_load_3d(out_s + cc * (BLOCK_M * 64), &tmC, bar(L::C_FULL), T.n0 + cc * 32, T.m0,
                          T.zd);
        }
      }
      named_bar_sync(1, 32 * NUM_PROMO_WARPS);
      // contiguous: padding blocks and rows (m_indices = -1) and bad experts are +0
      bool zero_row = MODE == kContiguous && T.skip != 0;
      if constexpr (MODE == kContiguous) {
        if (T.skip == 2 && ept == 0) raise_status(p, ST_EXPERT_RANGE);
        if (!T.skip) {
          const int id = __ldg(p.m_indices + T.m0 + row);
          if (id != T.e) {
            zero_row = true;
            if (id >= 0) raise_status(p, ST_EXPERT_RANGE);
          }
        }
      }
      bool c_in = false;
      if (has_c) {
        c_in = wait_bar(bar(L::C_FULL), cph, abort_flag, p);
        cph ^= 1;
      }
      const bool acc_in = !T.skip && wait_bar(bar(L::T_FULL + b), bph, abort_flag, p);
      __syncwarp();
      tc_fence_after();
#pragma unroll 1
      for (int c = c_lo; c < c_hi; ++c) {
        uint32_t v[32];
        if (acc_in) {
          tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(b * BN + c * 32), v);
          tmem_wait_ld(v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (c == c_hi - 1 && !T.skip) {
          // every tensor-memory load of this warp has completed: hand the
          // accumulator back (pair: on the leader's barrier)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PAIR && !leader) mbar_arrive_remote_relaxed(bar(L::T_EMPTY + b), 0);
            else mbar_arrive(bar(L::T_EMPTY + b));
          }
        }
        // staging: BN/32 chunks of [128 rows x 64 B], 64-byte swizzle (16-byte
        // unit u of row r at unit u ^ ((r >> 1) & 3)), as the store's tensor map expects
        const uint32_t rbase = out_s + c * (BLOCK_M * 64) + row * 64;
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const uint32_t addr = rbase + ((uu ^ ((row >> 1) & 3)) << 4);
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[uu * 8 + e]);
          if (c_in) {
            const uint4 cv = ld_shared_v4(addr);
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              f[2 * e] += __uint_as_float(cw[e] << 16);
              f[2 * e + 1] += __uint_as_float(cw[e] & 0xFFFF0000u);
            }
          }
          uint32_t w0 = pack_bf16x2(f[0], f[1]);
          uint32_t w1 = pack_bf16x2(f[2], f[3]);
          uint32_t w2 = pack_bf16x2(f[4], f[5]);
          uint32_t w3 = pack_bf16x2(f[6], f[7]);
          if (zero_row) w0 = w1 = w2 = w3 = 0u;
          st_shared_v4(addr, w0, w1, w2, w3);
        }
      }
      if (!T.skip) {
        if (++b == NACC) { b = 0; bph ^= 1; }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 32 * NUM_PROMO_WARPS);
      if (MODE != kMasked || T.rows == BLOCK_M) {
        if (ept == 0 && !*abort_flag && T.rows > 0) {
          for (int cc = 0; cc < BN / 32; ++cc)
            if (T.n0 + cc * 32 < p.N)
              tma_store_3d(&tmD, out_s + cc * (BLOCK_M * 64), T.n0 + cc * 32, T.m0, T.zd);
          bulk_commit_group();
        }
      } else if (!*abort_flag) {
        // masked form, last tile of a group: rows >= masked_m[g] keep what D held
        constexpr int UPR = BN / 8;   // 16-byte units per row
        for (int i = ept; i < T.rows * UPR; i += 32 * NUM_PROMO_WARPS) {
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
    }
    if (ept == 0) bulk_wait_group0();
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

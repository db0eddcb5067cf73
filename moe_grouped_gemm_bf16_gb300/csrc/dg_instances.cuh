// Ahead-of-time kernel instances and their launch helpers.  Each instance is a
// fixed (BLOCK_N, stages, K split, form) combination of the kernel template;
// the host launcher picks one per call.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "dg_params.h"

namespace dgk {

struct Maps {
  CUtensorMap a, b, sa, d, c;  // c: the dense form's addend (unused when there is none)
};

struct Instance {
  int block_n;
  int stages;
  int split;  // 1: may run as a cluster with the K groups split across its CTAs
  int mode;
  int a_rows;      // rows of A per tile loaded by TMA (128, or 64 for M <= 64)
  int pair;        // 1: CTA-pair form (cta_group::2, 256-row tiles over a 2-CTA cluster)
  int layout;      // operand storage (kNT, kNN, kTN, kTT)
  int sfp;         // 1: packed UE8M0 scales
  int bs;          // block-scaled MMA (the tensor cores apply the UE8M0 scales; no promotion):
                   // 0 no, else the number of MMA issuers (1 or 2)
  int nacc;        // block-scaled: tensor-memory accumulators (tiles in flight)
  int fixed_smem;  // shared memory that does not depend on the shape (bytes)
  cudaError_t (*launch)(const Maps& m, const Params& p, int grid, int cluster, int smem,
                        cudaStream_t s);
  cudaError_t (*set_smem)(int smem);
  cudaError_t (*max_clusters)(int cluster, int smem, int* out);
};

// Per-form instance tables (defined in dg_inst_*.cu).
const Instance* instances_dense(int* count);
const Instance* instances_contiguous(int* count);
const Instance* instances_masked(int* count);
// dense nn / tn / tt and the K-grouped tn form (MN-major operands)
const Instance* instances_mn(int* count);
// the same tables with packed UE8M0 scales
const Instance* instances_dense_ue8m0(int* count);
const Instance* instances_contiguous_ue8m0(int* count);
const Instance* instances_masked_ue8m0(int* count);
const Instance* instances_mn_ue8m0(int* count);
// block-scaled instances for packed UE8M0 scales (defined in dg_inst_bs*.cu)
const Instance* instances_bs_dense(int* count);
const Instance* instances_bs_contiguous(int* count);
const Instance* instances_bs_masked(int* count);
const Instance* instances_bs_mn(int* count);

}  // namespace dgk

#ifdef DGK_DEFINE_INSTANCES
#include "dg_kernel.cuh"

namespace dgk {

template <int BN, int STAGES, bool SPLIT, int MODE, int AROWS = BLOCK_M, bool PAIR = false,
          int LAYOUT = kNT, bool SFP = false>
struct InstanceOf {
  static constexpr auto kernel =
      fp8_gemm_kernel<BN, STAGES, SPLIT, MODE, AROWS, PAIR, LAYOUT, SFP>;

  static cudaError_t launch(const Maps& m, const Params& p, int grid, int cluster, int smem,
                            cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    // programmatic dependent launch: the prologue may overlap the previous
    // kernel in the stream; the kernel waits for it before reading memory
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (SPLIT || PAIR) {
      attr[n].id = cudaLaunchAttributeClusterDimension;
      attr[n].val.clusterDim.x = cluster;
      attr[n].val.clusterDim.y = 1;
      attr[n].val.clusterDim.z = 1;
      ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, m.a, m.b, m.sa, m.d, m.c, p);
  }

  static cudaError_t set_smem(int smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  }

  static cudaError_t max_clusters(int cluster, int smem, int* out) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kernel, &cfg);
  }

  static Instance make() {
    return Instance{BN, STAGES, SPLIT ? 1 : 0, MODE, AROWS, PAIR ? 1 : 0, LAYOUT, SFP ? 1 : 0,
                    0, 0, SmemLayout<BN, STAGES, SPLIT, AROWS, PAIR>::DYN_OFF + 1024, &launch,
                    &set_smem, &max_clusters};
  }
};

}  // namespace dgk
#endif

#ifdef DGK_DEFINE_BS_INSTANCES
#include "dg_kernel_bs.cuh"

namespace dgk {

// A block-scaled instance: the same launch interface as InstanceOf.
template <int BN, int STAGES, int MODE, bool PAIR, int NACC, int LAYOUT = kNT, int ISS = 1>
struct BsInstanceOf {
  static constexpr auto kernel = fp8_gemm_bs_kernel<BN, STAGES, MODE, PAIR, NACC, LAYOUT, ISS>;

  static cudaError_t launch(const Maps& m, const Params& p, int grid, int cluster, int smem,
                            cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(BS_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (PAIR) {
      attr[n].id = cudaLaunchAttributeClusterDimension;
      attr[n].val.clusterDim.x = cluster;
      attr[n].val.clusterDim.y = 1;
      attr[n].val.clusterDim.z = 1;
      ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, m.a, m.b, m.sa, m.d, m.c, p);
  }

  static cudaError_t set_smem(int smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  }

  static cudaError_t max_clusters(int cluster, int smem, int* out) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(BS_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kernel, &cfg);
  }

  static Instance make() {
    return Instance{BN, STAGES, 0, MODE, BLOCK_M, PAIR ? 1 : 0, LAYOUT, 1, ISS, NACC,
                    BsLayout<BN, STAGES, PAIR, NACC, ISS>::DYN_OFF + 1024, &launch, &set_smem,
                    &max_clusters};
  }
};

}  // namespace dgk
#endif

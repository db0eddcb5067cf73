// Per-token 1x128 FP8 activation quantiser: the step that produces the GEMMs'
// left operand A (e4m3) and its scales sa (fp32, K-group-major, as the GEMMs
// read them: es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de
// layout").  For each row m and 128-wide K group g of a bf16 matrix X:
//
//   a        = max(max_k |X[m,k]|, 1e-4)
//   sa[g][m] = a / 448
//   Q[m,k]   = e4m3, round to nearest even, saturating (X[m,k] * (448 / a))
//
// all in fp32 (two divisions per group, one multiply per element).
//
// UE8M0 form (the scale format of the SM100 kernels, same page and section:
// packed UE8M0, four per 32-bit word): the scale is rounded up to a power of
// two, s = the smallest 2^e >= fp32(a / 448), so x / s is exact; the byte
// 127 + e goes to byte g % 4 of word [g / 4][m] of the packed scales.
//
// Memory-bound (3 bytes per element plus 4 per group), so the instruction
// count per byte is what to keep low: the grid is (row blocks, K groups,
// batch), so a thread finds its row and group without a division; 8 threads
// take one (row, group) unit, 16 elements each (two 16-byte loads, one 16-byte
// store), and a warp covers 4 consecutive rows of one group; the group maximum
// is a 3-step shuffle reduction within the 8 lanes.  A block covers 32 rows per
// pass and QT_ROWS passes, whose loads are all in flight before any is used.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_quant.h"

namespace dgk {
namespace {

constexpr int QT_THREADS = 256;  // 8 warps x 4 rows = 32 rows per pass
constexpr int QT_ROWS = 2;       // passes (rows per thread)

// two fp32 -> two e4m3 codes (round to nearest even, saturating to +-448),
// `lo` in the low byte
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <bool UE8M0>
__global__ void __launch_bounds__(QT_THREADS)
quantize_1x128_kernel(const uint4* __restrict__ X, uint4* __restrict__ Q, float* __restrict__ sa,
                      int M, int K, int kb, int ld_sa) {
  // launched with programmatic dependent launch: the inputs may come from the
  // previous kernel in the stream, so nothing is read before it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;                                   // 16-element slice of the group
  const int row0 = blockIdx.x * (32 * QT_ROWS) + (threadIdx.x >> 5) * 4 + (lane >> 3);
  const int g = blockIdx.y;
  const int z = blockIdx.z;
  uint4 v[QT_ROWS][2];
  size_t off[QT_ROWS];  // offset of this thread's 16 elements, in 16-element units
#pragma unroll
  for (int j = 0; j < QT_ROWS; ++j) {
    const int m = row0 + j * 32;
    off[j] = ((static_cast<size_t>(z) * M + m) * K + static_cast<size_t>(g) * 128) / 16 + sub;
    v[j][0] = v[j][1] = make_uint4(0, 0, 0, 0);
    if (m < M) {
      v[j][0] = ld_stream_v4(X + 2 * off[j]);
      v[j][1] = ld_stream_v4(X + 2 * off[j] + 1);
    }
  }
#pragma unroll
  for (int j = 0; j < QT_ROWS; ++j) {
    const int m = row0 + j * 32;
    float x[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      x[8 * h + 0] = bf16_lo(v[j][h].x); x[8 * h + 1] = bf16_hi(v[j][h].x);
      x[8 * h + 2] = bf16_lo(v[j][h].y); x[8 * h + 3] = bf16_hi(v[j][h].y);
      x[8 * h + 4] = bf16_lo(v[j][h].z); x[8 * h + 5] = bf16_hi(v[j][h].z);
      x[8 * h + 6] = bf16_lo(v[j][h].w); x[8 * h + 7] = bf16_hi(v[j][h].w);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    // all 32 lanes take part (rows past M hold zeros); xor distances < 8 stay
    // within the unit's 8 lanes
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float a = fmaxf(amax, 1e-4f);
    float factor;
    uint32_t e8 = 0;   // UE8M0: the scale's exponent code
    if constexpr (UE8M0) {
      // t = a / 448 is a normal fp32 number here (a >= 1e-4, a <= bf16's largest);
      // its power-of-two ceiling is 2^(E - 127) when the mantissa is zero, else
      // 2^(E - 126), E the biased exponent; the factor 1 / s is exact
      const uint32_t tb = __float_as_uint(__fdiv_rn(a, 448.0f));
      e8 = ((tb >> 23) & 0xFFu) + ((tb & 0x7FFFFFu) != 0u ? 1u : 0u);
      factor = __uint_as_float((254u - e8) << 23);
    } else {
      factor = __fdiv_rn(448.0f, a);
    }
    uint4 w;
    w.x = cvt_e4m3x2(x[0] * factor, x[1] * factor) | (cvt_e4m3x2(x[2] * factor, x[3] * factor) << 16);
    w.y = cvt_e4m3x2(x[4] * factor, x[5] * factor) | (cvt_e4m3x2(x[6] * factor, x[7] * factor) << 16);
    w.z = cvt_e4m3x2(x[8] * factor, x[9] * factor) |
          (cvt_e4m3x2(x[10] * factor, x[11] * factor) << 16);
    w.w = cvt_e4m3x2(x[12] * factor, x[13] * factor) |
          (cvt_e4m3x2(x[14] * factor, x[15] * factor) << 16);
    if (m < M) {
      Q[off[j]] = w;
      if (sub == 0) {
        if constexpr (UE8M0) {
          // byte g % 4 of the packed word [z][g / 4][m] (little-endian)
          const int kbp = (kb + 3) >> 2;
          reinterpret_cast<uint8_t*>(sa)[((static_cast<size_t>(z) * kbp + (g >> 2)) * ld_sa + m) * 4 +
                                         (g & 3)] = static_cast<uint8_t>(e8);
        } else {
          sa[(static_cast<size_t>(z) * kb + g) * ld_sa + m] = __fdiv_rn(a, 448.0f);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize_1x128(const void* X, void* Q, float* sa, int num_groups, int M, int K,
                                  int ld_sa, int num_sms, cudaStream_t stream, bool ue8m0) {
  (void)num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + 32 * QT_ROWS - 1) / (32 * QT_ROWS), K / 128, num_groups);
  cfg.blockDim = dim3(QT_THREADS, 1, 1);
  cfg.stream = stream;
  // programmatic dependent launch: the blocks may be scheduled while the
  // previous kernel finishes; they wait for it before reading (griddepcontrol)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint4* Xv = static_cast<const uint4*>(X);
  uint4* Qv = static_cast<uint4*>(Q);
  return ue8m0 ? cudaLaunchKernelEx(&cfg, quantize_1x128_kernel<true>, Xv, Qv, sa, M, K, K / 128, ld_sa)
               : cudaLaunchKernelEx(&cfg, quantize_1x128_kernel<false>, Xv, Qv, sa, M, K, K / 128,
                                    ld_sa);
}

}  // namespace dgk

// Launcher of the per-token 1x128 FP8 activation quantiser (dg_quant.cu).
#pragma once
#include <cuda_runtime.h>

namespace dgk {

// X: bf16 [num_groups][M][K]; Q: e4m3 [num_groups][M][K];
// sa: fp32 [num_groups][K/128][ld_sa] (columns m < M written), or with
// `ue8m0` packed UE8M0 words [num_groups][ceil(K/512)][ld_sa] (the bytes of
// K groups < K/128 of columns m < M written).
// The caller has validated the arguments (K % 128 == 0, ld_sa >= M,
// num_groups * M * K/128 < 2^31, K/128 and num_groups <= 65535, 16-byte aligned
// X and Q).
cudaError_t launch_quantize_1x128(const void* X, void* Q, float* sa, int num_groups, int M, int K,
                                  int ld_sa, int num_sms, cudaStream_t stream, bool ue8m0 = false);

}  // namespace dgk

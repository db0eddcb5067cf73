// Block-scaled instances (packed UE8M0 scales applied by the tensor cores)
// with MN-major operands: dense nn / tn / tt and the K-grouped tn form.
#define DGK_DEFINE_BS_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_bs_mn(int* count) {
  static const Instance table[] = {
      BsInstanceOf<128, 6, kDense, false, 3, kNN>::make(),
      BsInstanceOf<256, 4, kDense, false, 1, kNN>::make(),
      BsInstanceOf<128, 6, kDense, false, 3, kTN>::make(),
      BsInstanceOf<256, 4, kDense, false, 1, kTN>::make(),
      BsInstanceOf<128, 6, kDense, false, 3, kTT>::make(),
      BsInstanceOf<256, 4, kDense, false, 1, kTT>::make(),
      BsInstanceOf<128, 6, kKGrouped, false, 3, kTN>::make(),
      BsInstanceOf<256, 4, kKGrouped, false, 1, kTN>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

// MN-major instances (nn / tn / tt and K-grouped) with packed UE8M0 scales.
#define DGK_DEFINE_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_mn_ue8m0(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kDense, 128, false, kNN, true>::make(),
      InstanceOf<256, 3, false, kDense, 128, false, kNN, true>::make(),
      InstanceOf<128, 5, false, kDense, 128, false, kTN, true>::make(),
      InstanceOf<256, 3, false, kDense, 128, false, kTN, true>::make(),
      InstanceOf<128, 5, false, kDense, 128, false, kTT, true>::make(),
      InstanceOf<256, 3, false, kDense, 128, false, kTT, true>::make(),
      InstanceOf<128, 6, true, kDense, 128, false, kNN, true>::make(),
      InstanceOf<128, 6, true, kDense, 128, false, kTN, true>::make(),
      InstanceOf<128, 6, true, kDense, 128, false, kTT, true>::make(),
      InstanceOf<128, 5, false, kKGrouped, 128, false, kTN, true>::make(),
      InstanceOf<256, 3, false, kKGrouped, 128, false, kTN, true>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

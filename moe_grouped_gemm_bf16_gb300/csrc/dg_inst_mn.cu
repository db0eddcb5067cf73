// Instances with MN-major operands: the dense nn / tn / tt layouts and the
// K-grouped tn form (A stored [K][M], B stored [K][N]).
#define DGK_DEFINE_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_mn(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kDense, 128, false, kNN>::make(),
      InstanceOf<256, 3, false, kDense, 128, false, kNN>::make(),
      InstanceOf<128, 5, false, kDense, 128, false, kTN>::make(),
      InstanceOf<256, 3, false, kDense, 128, false, kTN>::make(),
      InstanceOf<128, 5, false, kDense, 128, false, kTT>::make(),
      InstanceOf<256, 3, false, kDense, 128, false, kTT>::make(),
      // K split over a cluster (decode shapes; an MN-major A is always a full 128-row box)
      InstanceOf<128, 6, true, kDense, 128, false, kNN>::make(),
      InstanceOf<128, 6, true, kDense, 128, false, kTN>::make(),
      InstanceOf<128, 6, true, kDense, 128, false, kTT>::make(),
      InstanceOf<128, 5, false, kKGrouped, 128, false, kTN>::make(),
      InstanceOf<256, 3, false, kKGrouped, 128, false, kTN>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

// Dense-form kernel instances.
#define DGK_DEFINE_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_dense(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kDense>::make(),
      InstanceOf<256, 3, false, kDense>::make(),
      InstanceOf<128, 6, true, kDense>::make(),
      InstanceOf<128, 8, true, kDense, 64>::make(),
      InstanceOf<256, 5, true, kDense, 64>::make(),
      InstanceOf<256, 4, false, kDense, 128, true>::make(),
      InstanceOf<128, 6, false, kDense, 128, true>::make(),
      InstanceOf<64, 8, false, kDense>::make(),
      InstanceOf<64, 8, true, kDense>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

// Contiguous M-grouped kernel instances.
#define DGK_DEFINE_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_contiguous(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kContiguous>::make(),
      InstanceOf<256, 3, false, kContiguous>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

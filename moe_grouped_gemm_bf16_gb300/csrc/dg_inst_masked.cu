// Masked M-grouped kernel instances.
#define DGK_DEFINE_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_masked(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kMasked>::make(),
      InstanceOf<256, 3, false, kMasked>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

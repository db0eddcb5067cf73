// Masked M-grouped kernel instances.
#define DGK_DEFINE_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_masked(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kMasked>::make(),
      InstanceOf<256, 3, false, kMasked>::make(),
      InstanceOf<64, 8, false, kMasked>::make(),
      // CTA pairs: 256-row M blocks, each CTA loading half of the B tile
      InstanceOf<256, 4, false, kMasked, 128, true>::make(),
      InstanceOf<128, 6, false, kMasked, 128, true>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

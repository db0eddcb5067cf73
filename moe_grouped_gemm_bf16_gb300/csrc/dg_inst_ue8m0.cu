// Dense, contiguous and masked instances with packed UE8M0 scales (the same
// configurations as the fp32-scale tables).
#define DGK_DEFINE_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_dense_ue8m0(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kDense, 128, false, kNT, true>::make(),
      InstanceOf<256, 3, false, kDense, 128, false, kNT, true>::make(),
      InstanceOf<128, 6, true, kDense, 128, false, kNT, true>::make(),
      InstanceOf<128, 8, true, kDense, 64, false, kNT, true>::make(),
      InstanceOf<256, 5, true, kDense, 64, false, kNT, true>::make(),
      InstanceOf<256, 4, false, kDense, 128, true, kNT, true>::make(),
      InstanceOf<128, 6, false, kDense, 128, true, kNT, true>::make(),
      InstanceOf<64, 8, false, kDense, 128, false, kNT, true>::make(),
      InstanceOf<64, 8, true, kDense, 128, false, kNT, true>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}

const Instance* instances_contiguous_ue8m0(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kContiguous, 128, false, kNT, true>::make(),
      InstanceOf<256, 3, false, kContiguous, 128, false, kNT, true>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}

const Instance* instances_masked_ue8m0(int* count) {
  static const Instance table[] = {
      InstanceOf<128, 5, false, kMasked, 128, false, kNT, true>::make(),
      InstanceOf<256, 3, false, kMasked, 128, false, kNT, true>::make(),
      InstanceOf<64, 8, false, kMasked, 128, false, kNT, true>::make(),
      InstanceOf<256, 4, false, kMasked, 128, true, kNT, true>::make(),
      InstanceOf<128, 6, false, kMasked, 128, true, kNT, true>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

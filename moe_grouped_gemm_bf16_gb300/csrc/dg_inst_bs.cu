// Block-scaled instances (packed UE8M0 scales applied by the tensor cores):
// dense, contiguous and masked nt forms.  (BN, stages, form, CTA pair,
// accumulators in tensor memory); the stage counts fill the 227 KB of shared
// memory next to the two 8 KB staging buffers of the epilogue.
#define DGK_DEFINE_BS_INSTANCES
#include "dg_instances.cuh"

namespace dgk {
const Instance* instances_bs_dense(int* count) {
  static const Instance table[] = {
      BsInstanceOf<128, 6, kDense, false, 3>::make(),
      BsInstanceOf<224, 4, kDense, false, 2>::make(),
      BsInstanceOf<256, 4, kDense, false, 1>::make(),
      BsInstanceOf<256, 6, kDense, true, 1>::make(),
      BsInstanceOf<128, 8, kDense, true, 3>::make(),
      BsInstanceOf<224, 4, kDense, false, 1, kNT, 2>::make(),
      BsInstanceOf<224, 6, kDense, true, 1, kNT, 2>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}

const Instance* instances_bs_contiguous(int* count) {
  static const Instance table[] = {
      BsInstanceOf<128, 6, kContiguous, false, 3>::make(),
      BsInstanceOf<224, 4, kContiguous, false, 2>::make(),
      BsInstanceOf<256, 4, kContiguous, false, 1>::make(),
      BsInstanceOf<224, 4, kContiguous, false, 1, kNT, 2>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}

const Instance* instances_bs_masked(int* count) {
  static const Instance table[] = {
      BsInstanceOf<128, 6, kMasked, false, 3>::make(),
      BsInstanceOf<256, 4, kMasked, false, 1>::make(),
      BsInstanceOf<256, 6, kMasked, true, 1>::make(),
      BsInstanceOf<128, 8, kMasked, true, 3>::make(),
      BsInstanceOf<224, 4, kMasked, false, 1, kNT, 2>::make(),
      BsInstanceOf<224, 6, kMasked, true, 1, kNT, 2>::make(),
  };
  *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}
}  // namespace dgk

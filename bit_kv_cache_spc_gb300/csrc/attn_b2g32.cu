// The attention kernels at 2 bits and group size 32 (see attention.cuh).
#include "attention.cuh"

namespace spc {
const AttnVariant& attn_variant_b2g32() {
  static const AttnVariant v = AttnVariantImpl<2, 32>::table();
  return v;
}
}  // namespace spc

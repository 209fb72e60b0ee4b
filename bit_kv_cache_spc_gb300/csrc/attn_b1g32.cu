// The attention kernels at 1 bit and group size 32 (see attention.cuh).
#include "attention.cuh"

namespace spc {
const AttnVariant& attn_variant_b1g32() {
  static const AttnVariant v = AttnVariantImpl<1, 32>::table();
  return v;
}
}  // namespace spc

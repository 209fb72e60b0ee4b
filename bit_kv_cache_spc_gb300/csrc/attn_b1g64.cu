// The attention kernels at 1 bit and group size 64 (see attention.cuh).
#include "attention.cuh"

namespace spc {
const AttnVariant& attn_variant_b1g64() {
  static const AttnVariant v = AttnVariantImpl<1, 64>::table();
  return v;
}
}  // namespace spc

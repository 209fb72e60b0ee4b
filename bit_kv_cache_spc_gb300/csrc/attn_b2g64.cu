// The attention kernels at 2 bits and group size 64 (see attention.cuh).
#include "attention.cuh"

namespace spc {
const AttnVariant& attn_variant_b2g64() {
  static const AttnVariant v = AttnVariantImpl<2, 64>::table();
  return v;
}
}  // namespace spc

// decode_split_masked.cu -- K3+K4 with a boolean or additive attention mask (the kernel
// itself is in decode_split.cuh; a separate translation unit so both sets compile in
// parallel).
#include "decode_split.cuh"

namespace gqa {

gqa_status launch_decode_split_masked(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  if (c.Dv != c.p.head_dim) return launch_decode_split_vdim(c, dp, wl);  // its own translation unit
  return launch_decode_split_impl<true, false>(c, dp, wl);
}

}  // namespace gqa

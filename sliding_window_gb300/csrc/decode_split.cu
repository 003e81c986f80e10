// decode_split.cu -- K3+K4: the split-KV decode kernels without an attention mask (the
// kernel itself is in decode_split.cuh).
#include "decode_split.cuh"

namespace gqa {

gqa_status launch_decode_split(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  if (c.Dv != c.p.head_dim) return launch_decode_split_vdim(c, dp, wl);  // its own translation unit
  return launch_decode_split_impl<false, false>(c, dp, wl);
}

}  // namespace gqa

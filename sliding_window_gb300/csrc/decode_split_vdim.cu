// decode_split_vdim.cu -- K3+K4 for a V head dimension that differs from the Q/K one
// (onnx-light-cpu "Attention Kernel Design", "Layouts and semantics"), with or without an
// attention mask (the kernel itself is in decode_split.cuh).
#include "decode_split.cuh"

namespace gqa {

gqa_status launch_decode_split_vdim(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  return c.mask ? launch_decode_split_impl<true, true>(c, dp, wl) : launch_decode_split_impl<false, true>(c, dp, wl);
}

}  // namespace gqa

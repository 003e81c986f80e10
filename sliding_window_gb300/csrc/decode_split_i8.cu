// decode_split_i8.cu -- K3+K4 over an int8 KV cache with one scale per kv head for K and
// V (the kernel itself is in decode_split.cuh).
#include "decode_split.cuh"

namespace gqa {

gqa_status launch_decode_split_i8(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  return launch_decode_split_impl<false, false, true, true>(c, dp, wl);
}

}  // namespace gqa

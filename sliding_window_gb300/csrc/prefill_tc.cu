// prefill_tc.cu -- K2: the tensor-core prefill kernels without an attention mask (the
// kernel itself is in prefill_tc.cuh).
#include "prefill_tc.cuh"

namespace gqa {

gqa_status launch_prefill_tc(const Call &c) {
  if (c.Dv != c.p.head_dim) return launch_prefill_tc_vdim(c);  // its own translation unit
  return launch_prefill_tc_any<0, false>(c);
}

}  // namespace gqa

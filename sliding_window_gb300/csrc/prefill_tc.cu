// prefill_tc.cu -- K2: the tensor-core prefill kernels without an attention mask (the
// kernel itself is in prefill_tc.cuh).
#include "prefill_tc.cuh"

namespace gqa {

gqa_status launch_prefill_tc(const Call &c) { return launch_prefill_tc_any<0>(c); }

}  // namespace gqa

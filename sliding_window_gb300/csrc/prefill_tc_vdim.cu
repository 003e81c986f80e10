// prefill_tc_vdim.cu -- K2 for a V head dimension that differs from the Q/K one
// (onnx-light-cpu "Attention Kernel Design", "Layouts and semantics"); the kernel itself is
// in prefill_tc.cuh.  Masked prefill with such a V runs on the CUDA-core kernel.
#include "prefill_tc.cuh"

namespace gqa {

gqa_status launch_prefill_tc_vdim(const Call &c) { return launch_prefill_tc_any<0, true>(c); }

}  // namespace gqa

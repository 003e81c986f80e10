// prefill_tc_masked.cu -- K2 with a boolean (MK = 1) or additive (MK = 2) attention mask
// staged by TMA (the kernel itself is in prefill_tc.cuh; a separate translation unit so the
// sets compile in parallel and the unmasked kernels keep their registers).
#include "prefill_tc.cuh"

namespace gqa {

gqa_status launch_prefill_tc_masked(const Call &c) {
  if (c.mask_kind == GQA_MASK_KEEP) return launch_prefill_tc_any<1, false>(c);
  // a head-broadcast additive mask is staged once for both heads of a CTA (MK 3), which
  // leaves the K ring its two stages
  if (c.mask_kind == GQA_MASK_ADD) return c.mask_sh == 0 ? launch_prefill_tc_any<3, false>(c) : launch_prefill_tc_any<2, false>(c);
  return GQA_ERR_INVALID_ARG;
}

}  // namespace gqa

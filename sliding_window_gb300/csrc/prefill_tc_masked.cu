// prefill_tc_masked.cu -- K2 with a boolean (MK = 1) or additive (MK = 2) attention mask
// staged by TMA (the kernel itself is in prefill_tc.cuh; a separate translation unit so the
// sets compile in parallel and the unmasked kernels keep their registers).
#include "prefill_tc.cuh"

namespace gqa {
namespace {

// The block map of a boolean mask ([P4] "Compute paths": a block the mask removes entirely
// is skipped).  One CTA per (128-row query tile, q head, batch) of the mask's shape (a
// broadcast dimension has extent 1); bit c of word w is set when any of the tile's rows
// keeps a key of 16-key chunk 32w + c.  Each warp reads whole rows, 16 bytes per lane.
__global__ void __launch_bounds__(256) mask_blockmap_kernel(const uint8_t *mask, long long sb, long long sh,
                                                            long long si, int q_len, int keys, int heads, int qtiles,
                                                            int words, uint32_t *map,
                                                            [[maybe_unused]] size_t map_extent,
                                                            [[maybe_unused]] int32_t *status) {
  const int qm = blockIdx.x, hm = blockIdx.y, bm = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = si == 0 ? 0 : qm * 128;
  const int nr = si == 0 ? 1 : min(128, q_len - r0);
  const uint8_t *base = mask + bm * sb + hm * sh;
  uint32_t *out = map + (((size_t)bm * heads + hm) * qtiles + qm) * words;
  const int nch = (keys + 15) / 16;
  __shared__ uint32_t part[8];
  for (int w = 0; w < words; ++w) {
    const int c = w * 32 + lane;
    bool any = false;
    if (c < nch) {
      for (int r = warp; r < nr && !any; r += 8) {
        const uint8_t *p = base + (r0 + r) * si + c * 16;
        if (c * 16 + 16 <= keys) {
          const uint4 v = *reinterpret_cast<const uint4 *>(p);
          any = (v.x | v.y | v.z | v.w) != 0u;
        } else {
          for (int k = 0; k < keys - c * 16; ++k) any |= p[k] != 0;
        }
      }
    }
    const uint32_t bits = __ballot_sync(0xffffffffu, any);
    if (lane == 0) part[warp] = bits;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t x = 0;
      for (int i = 0; i < 8; ++i) x |= part[i];
      GQA_GUARD((size_t)(out - map) + w, 1, map_extent, status)
      out[w] = x;
    }
    __syncthreads();
  }
}

}  // namespace

gqa_status launch_prefill_tc_masked(const Call &c) {
  if (c.mask_kind == GQA_MASK_KEEP) {
    if (c.blockmap) {
      const gqa_params &p = c.p;
      const int keys = c.mask_keys < p.cap_present ? c.mask_keys : p.cap_present;
      const int heads = c.mask_sh == 0 ? 1 : p.q_heads, qtiles = c.mask_si == 0 ? 1 : (p.q_len + 127) / 128;
      const int words = ((keys + 15) / 16 + 31) / 32;
      mask_blockmap_kernel<<<dim3(qtiles, heads, c.mask_sb == 0 ? 1 : p.batch), 256, 0, c.stream>>>(
          static_cast<const uint8_t *>(c.mask), c.mask_sb, c.mask_sh, c.mask_si, p.q_len, keys, heads, qtiles, words,
          c.blockmap, c.blockmap_extent, c.status);
      if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    }
    return launch_prefill_tc_any<1, false>(c);
  }
  // a head-broadcast additive mask is staged once for both heads of a CTA (MK 3), which
  // leaves the K ring its two stages
  if (c.mask_kind == GQA_MASK_ADD) return c.mask_sh == 0 ? launch_prefill_tc_any<3, false>(c) : launch_prefill_tc_any<2, false>(c);
  return GQA_ERR_INVALID_ARG;
}

}  // namespace gqa

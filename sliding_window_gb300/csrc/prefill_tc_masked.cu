// prefill_tc_masked.cu -- K2 with a boolean (MK = 1) or additive (MK = 2) attention mask
// staged by TMA (the kernel itself is in prefill_tc.cuh; a separate translation unit so the
// sets compile in parallel and the unmasked kernels keep their registers).
#include "prefill_tc.cuh"

namespace gqa {
namespace {

// The block map of a boolean mask ([P4] "Compute paths": a block the mask removes entirely
// is skipped).  Bit c of word w of row (b, h, query tile) is set when any of the tile's 128
// rows (one for a row-broadcast mask) keeps a key of 16-key chunk 32w + c.  One warp per
// word: lane l reads chunk 32w + l of every row (16 bytes, the rows' loads independent, so
// many are in flight), then the warp's ballot is the word.  grid (query tile x word group
// of 8, head, batch) of the mask's shape (a broadcast dimension has extent 1).
__global__ void __launch_bounds__(256) mask_blockmap_kernel(const uint8_t *mask, long long sb, long long sh,
                                                            long long si, int q_len, int keys, int heads, int qtiles,
                                                            int words, uint32_t *map,
                                                            [[maybe_unused]] size_t map_extent,
                                                            [[maybe_unused]] int32_t *status) {
  const int groups = (words + 7) / 8;
  const int qm = blockIdx.x / groups, w = (blockIdx.x % groups) * 8 + (int)(threadIdx.x >> 5);
  const int hm = blockIdx.y, bm = blockIdx.z, lane = threadIdx.x & 31;
  if (w >= words) return;
  const int r0 = si == 0 ? 0 : qm * 128;
  const int nr = si == 0 ? 1 : min(128, q_len - r0);
  const int c = w * 32 + lane, k0 = c * 16;
  const uint8_t *p = mask + bm * sb + hm * sh + r0 * si + k0;
  uint32_t any = 0;
  if (k0 + 16 <= keys) {
#pragma unroll 8
    for (int r = 0; r < nr; ++r) {
      const uint4 v = *reinterpret_cast<const uint4 *>(p + r * si);
      any |= v.x | v.y | v.z | v.w;
    }
  } else if (k0 < keys) {  // the last, partial chunk: only its keys
    for (int r = 0; r < nr; ++r)
      for (int k = 0; k < keys - k0; ++k) any |= p[r * si + k];
  }
  const uint32_t bits = __ballot_sync(0xffffffffu, any != 0u);
  if (lane == 0) {
    const size_t off = (((size_t)bm * heads + hm) * qtiles + qm) * words + w;
    GQA_GUARD(off, 1, map_extent, status)
    map[off] = bits;
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
      mask_blockmap_kernel<<<dim3(qtiles * ((words + 7) / 8), heads, c.mask_sb == 0 ? 1 : p.batch), 256, 0, c.stream>>>(
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

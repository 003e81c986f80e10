// launch.h -- host-side plan shared by the C-ABI entry points and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gqa.h"

#ifdef GQA_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace gqa {

// Tracing (-DGQA_NVTX, on in the bounds-checked debug build): every C-ABI call is one NVTX
// range named after the call, so that a profiler attributes the kernels it launches to it.
#ifdef GQA_NVTX
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
#define GQA_TRACE_CALL() ::gqa::NvtxRange gqa_trace_range_(__func__)
#else
#define GQA_TRACE_CALL()
#endif

// Element counts of the buffers a kernel writes (the bounds-checked debug build checks every
// store against them): out, present K and V (or their page pools), the rotated queries,
// and the workspace's partials, tickets and block map.
struct Extents {
  size_t out = 0, pk = 0, pv = 0, qrot = 0, part_acc = 0, part_ml = 0, tickets = 0, map = 0;
};

// One validated call: shapes and attributes plus every pointer the kernels need.
struct Call {
  gqa_params p;          // scale already resolved (0 -> 1/sqrt(D))
  int G = 1;             // q heads per kv head
  int esize = 2;         // bytes per element
  int Dv = 0;            // V head dim (v_head_dim, or head_dim when 0)
  const void *q = nullptr;        // query as it enters the scores (input q or q_rot)
  const void *q_in = nullptr;     // caller's q (before rotation)
  const void *k = nullptr, *v = nullptr;
  const void *past_k = nullptr, *past_v = nullptr;
  const int32_t *seqlens = nullptr;
  const int64_t *nonpad = nullptr;  // padded cache: valid keys per sequence (replaces seqlens)
  const void *cos = nullptr, *sin = nullptr;
  const float *head_sink = nullptr;
  void *out = nullptr;
  void *present_k = nullptr, *present_v = nullptr;
  void *q_rot = nullptr;           // where K1 writes rotated q (nullptr: not needed)
  int past_separate = 0;           // past and present are different buffers
  int append = 1;                  // 0: attention only (present already holds the step)
  // paged cache: present_k/v are pools [num_pages][Hkv][64][D], the table maps
  // (sequence, position / 64) to a page
  const int32_t *block_table = nullptr;
  int max_pages = 0, num_pages = 0;
  // attention mask: element [b][hq][i][key] at b*mask_sb + hq*mask_sh + i*mask_si + key,
  // kind 1 = uint8 keep flags, 2 = additive values of the dtype; keys < mask_keys
  const void *mask = nullptr;
  int mask_kind = 0, mask_keys = 0;
  long long mask_sb = 0, mask_sh = 0, mask_si = 0;
  // boolean mask on the tensor-core prefill: room for its block map in the workspace, or null
  uint32_t *blockmap = nullptr;
  size_t blockmap_extent = 0;  // its words
  // f8 cache: present_k/v hold E4M3 codes; the stored value is code * scale of the kv head
  int q8 = 0;  // one-byte cache codes: 1 E4M3, 2 int8
  const float *k_scale = nullptr, *v_scale = nullptr;
  int32_t *status = nullptr;
  // failure-path test hook (gqa_test_stall_waits): the limit of the kernels' pipeline waits
  // in SM cycles (0: the kernels' default), and whether their first wait is on a barrier
  // that nothing completes
  long long wait_limit = 0;
  int stall = 0;
  cudaStream_t stream = nullptr;
  char *ws = nullptr;
  size_t ws_bytes = 0;
};

// Split-KV decode plan.  The visible band of each (b, kv head) group is cut into `splits`
// equal chunks (one CTA each).  The plan depends on the params and the GPU's SM count; the
// workspace is sized for the largest plan any GPU of up to kPlanMaxSms SMs could choose, so
// that it depends on the params only.
constexpr int kDecodeMaxSplits = 64;
constexpr int kDecodeMaxCluster = 8;  // portable cluster size
constexpr int kPlanMaxSms = 512;
struct DecodePlan {
  bool eligible = false;  // the split kernel handles these params
  int rows = 0;           // R = G * curr query rows per CTA
  int mtiles = 0;         // ceil(R / 16)
  int splits = 1;         // chunks per group
  bool cluster = false;   // 2..8 chunks: one cluster per group, combined in shared memory
};

struct WsLayout {
  size_t q_rot_off = 0, q_rot_bytes = 0;
  size_t part_acc_off = 0, part_acc_bytes = 0;
  size_t part_ml_off = 0, part_ml_bytes = 0;
  size_t tickets_off = 0, tickets_bytes = 0;
  size_t blockmap_off = 0, blockmap_bytes = 0;  // a boolean mask's block map (tensor-core prefill)
  size_t total = 0;
};

// sms: the SM count of the GPU that runs the kernel (device_sm_count()), or kPlanMaxSms for
// the upper bound that sizes the workspace.
DecodePlan decode_plan(const gqa_params &p, int sms);
WsLayout workspace_layout(const gqa_params &p, bool need_q_rot);

// The element counts of a call's buffers (the bounds-checked debug build).
inline Extents extents_of(const Call &c, const WsLayout &wl) {
  Extents e;
  const gqa_params &p = c.p;
  e.out = (size_t)p.batch * p.q_len * p.q_heads * c.Dv;
  const size_t rows = c.block_table ? (size_t)c.num_pages * p.kv_heads * 64 : (size_t)p.batch * p.kv_heads * p.cap_present;
  e.pk = rows * p.head_dim;
  e.pv = rows * c.Dv;
  e.qrot = c.q_rot ? (size_t)p.batch * p.q_len * p.q_heads * p.head_dim : 0;
  if (c.ws) {
    e.part_acc = wl.part_acc_bytes / 4;
    e.part_ml = wl.part_ml_bytes / 4;
    e.tickets = wl.tickets_bytes / 4;
    e.map = wl.blockmap_bytes / 4;
  }
  return e;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda link).
// 3D map over a [outer, mid, inner] tensor of 16-bit elements with a 128B-swizzled box of
// {64, box_mid, 1}.  Returns false on failure.
bool encode_kv_map(CUtensorMap *map, const void *base, int inner, int mid, long long outer, int box_mid,
                   int esize);
// 4D map over the same [outer, rows, D] tensor of 16-bit elements whose single box of
// box_rows rows lands as [D/64][box_rows][64 columns], 128B-swizzled: one copy per tile.
bool encode_kv_tile_map(CUtensorMap *map, const void *base, int D, int rows, long long outer, int box_rows,
                        int esize);
// 3D map over an f8 cache [outer, rows, inner] of bytes (inner <= 128): box {inner, box_rows,
// 1}, 128B-swizzled rows.
bool encode_kv8_map(CUtensorMap *map, const void *base, int inner, int rows, long long outer, int box_rows);
// 4D map over q laid out [B, L, H, D]: box {64, 1, box_rows, 1}, 128B swizzle.
bool encode_q_map(CUtensorMap *map, const void *base, int D, int H, int L, int B, int box_rows, int esize);

// 4D map over an attention mask [B][H][I][keys] of 1- or 2-byte elements with byte strides
// (0 = broadcast dimension): box {box_keys, box_rows, 1, 1}, 128B swizzle.
bool encode_mask_map(CUtensorMap *map, const void *base, int keys, int I, int H, int B, long long si_bytes,
                     long long sh_bytes, long long sb_bytes, int box_keys, int box_rows, int esize);

int device_sm_count();

gqa_status launch_rope_append(const Call &c);
gqa_status launch_copy_past(const Call &c);  // rows [0, past_b) of past into present only
gqa_status launch_attention_simt(const Call &c);
gqa_status launch_decode_split(const Call &c, const DecodePlan &dp, const WsLayout &wl);
gqa_status launch_decode_split_masked(const Call &c, const DecodePlan &dp, const WsLayout &wl);
gqa_status launch_decode_split_vdim(const Call &c, const DecodePlan &dp, const WsLayout &wl);  // Dv != D
gqa_status launch_decode_split_q8(const Call &c, const DecodePlan &dp, const WsLayout &wl);    // f8 cache, D = Dv = 128
gqa_status launch_decode_split_i8(const Call &c, const DecodePlan &dp, const WsLayout &wl);    // int8 cache, D = Dv = 128
gqa_status launch_prefill_tc(const Call &c);
gqa_status launch_prefill_tc_masked(const Call &c);  // c.mask set: kind 1 or 2
gqa_status launch_prefill_tc_vdim(const Call &c);    // Dv != D, no mask

}  // namespace gqa

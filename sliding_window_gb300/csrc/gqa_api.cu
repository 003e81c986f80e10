// gqa_api.cu -- the C ABI of libgqa: host-side validation, planning and kernel launches.
//
// onnx-light-cpu "Attention Kernel Design", "Descriptor and invocation plan": attributes
// and wiring are validated first, then a light plan (layouts, strides, head mapping,
// total KV length) is rebuilt for every invocation; "Scheduling, precision, and
// invariants": head counts positive and divisible, matching types, invalid pairings fail
// explicitly.  Nothing here allocates memory or synchronizes the device.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gqa.h"
#include "launch.h"
#ifdef GQA_BOUNDS_CHECK
#include "common.cuh"
#endif

namespace gqa {
namespace {

constexpr size_t kAlign = 256;
// failure-path test hook (gqa_test_stall_waits): 0, or the SM cycles after which the kernels'
// pipeline waits give up, their first wait being on a barrier that nothing completes
std::atomic<long long> g_test_stall{0};
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-checkable validity of the params alone (no pointers).
gqa_status check_params(const gqa_params *p) {
  if (!p) return GQA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->q_heads < 1 || p->kv_heads < 1 || p->q_len < 1) return GQA_ERR_INVALID_ARG;
  if (p->q_heads % p->kv_heads != 0) return GQA_ERR_INVALID_ARG;
  if (p->dtype != GQA_F32 && p->dtype != GQA_F16 && p->dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (!(p->scale >= 0.f) || !isfinite(p->scale)) return GQA_ERR_INVALID_ARG;
  if (!(p->softcap >= 0.f) || !isfinite(p->softcap)) return GQA_ERR_INVALID_ARG;
  if (p->window != -1 && p->window < 1) return GQA_ERR_INVALID_ARG;
  if ((p->causal | 1) != 1 || (p->do_rotary | 1) != 1 || (p->smooth_softmax | 1) != 1) return GQA_ERR_INVALID_ARG;
  if ((p->rotary_interleaved | 1) != 1 || (p->kv_ring | 1) != 1) return GQA_ERR_INVALID_ARG;
  if (p->rotary_interleaved) return GQA_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return GQA_ERR_UNSUPPORTED;
  if (p->v_head_dim < 0) return GQA_ERR_INVALID_ARG;
  if (p->v_head_dim != 0 && p->v_head_dim != 64 && p->v_head_dim != 128) return GQA_ERR_UNSUPPORTED;
  if (p->kv_ring && p->v_head_dim != 0 && p->v_head_dim != p->head_dim) return GQA_ERR_UNSUPPORTED;
  if (p->cap_present < p->q_len || p->cap_past < 0) return GQA_ERR_CAPACITY;
  if (p->do_rotary && p->rope_len < 1) return GQA_ERR_INVALID_ARG;
  if (p->kv_ring) {  // position p in slot p % cap: every key the step sees must still be resident
    if (p->window < 1) return GQA_ERR_INVALID_ARG;
    if ((long long)p->window + p->q_len - 1 > p->cap_present) return GQA_ERR_CAPACITY;
    if (p->cap_present % 64 != 0) return GQA_ERR_UNSUPPORTED;  // 64-key tiles never straddle the wrap
  }
  // TMA coordinates and the kernels' index arithmetic are 32-bit per dimension
  const long long rows = (long long)p->batch * p->kv_heads;
  if (rows > (1ll << 30) || (long long)p->q_len * p->q_heads > (1ll << 30)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool encode_kv_map(CUtensorMap *map, const void *base, int inner, int mid, long long outer, int box_mid, int esize) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)inner * esize, (cuuint64_t)inner * esize * mid};
  cuuint32_t box[3] = {64, (cuuint32_t)box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                  const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_kv_tile_map(CUtensorMap *map, const void *base, int D, int rows, long long outer, int box_rows,
                        int esize) {
  auto fn = encode_fn();
  if (!fn) return false;
  // dims (64 columns, row, 64-column half, group): strides need not increase, so one box
  // {64, box_rows, D/64, 1} lands as [half][row][64 columns], the same image as D/64
  // separate 3D boxes of 64 columns
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(D / 64), (cuuint64_t)outer};
  cuuint64_t strides[3] = {(cuuint64_t)D * esize, (cuuint64_t)64 * esize, (cuuint64_t)rows * D * esize};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)(D / 64), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_kv8_map(CUtensorMap *map, const void *base, int inner, int rows, long long outer, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)inner * rows};
  cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap *map, const void *base, int D, int H, int L, int B, int box_rows, int esize) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * esize, (cuuint64_t)D * esize * H, (cuuint64_t)D * esize * H * L};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                  const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_mask_map(CUtensorMap *map, const void *base, int keys, int I, int H, int B, long long si_bytes,
                     long long sh_bytes, long long sb_bytes, int box_keys, int box_rows, int esize) {
  auto fn = encode_fn();
  if (!fn) return false;
  // a broadcast dimension (stride 0) becomes an extent of 1 read at coordinate 0, with the
  // packed stride it would have had (never used)
  const cuuint64_t row = ((cuuint64_t)keys * esize + 15) / 16 * 16;
  cuuint64_t dims[4] = {(cuuint64_t)keys, (cuuint64_t)(si_bytes ? I : 1), (cuuint64_t)(sh_bytes ? H : 1),
                        (cuuint64_t)(sb_bytes ? B : 1)};
  cuuint64_t strides[3];
  strides[0] = si_bytes ? (cuuint64_t)si_bytes : row;
  strides[1] = sh_bytes ? (cuuint64_t)sh_bytes : strides[0] * dims[1];
  strides[2] = sb_bytes ? (cuuint64_t)sb_bytes : strides[1] * dims[2];
  cuuint32_t box[4] = {(cuuint32_t)box_keys, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                  const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

DecodePlan decode_plan(const gqa_params &p, int sms) {
  DecodePlan d;
  const int G = p.q_heads / p.kv_heads;
  d.rows = G * p.q_len;
  d.mtiles = (d.rows + 15) / 16;
  const int dv = p.v_head_dim ? p.v_head_dim : p.head_dim;
  d.eligible = p.dtype != GQA_F32 &&
               (dv != p.head_dim ? d.mtiles <= 2  // different V head dim: up to 32 rows per group
                                 : (p.head_dim == 128 && d.mtiles <= 2) || (p.head_dim == 64 && d.mtiles <= 4));
  if (sms < 1) sms = 1;
  // longest visible band of one group: [max(0, past - W + 1), past + curr)
  long long lmax = p.cap_present;
  if (p.window > 0) lmax = std::min<long long>(lmax, (long long)p.window + p.q_len - 1);
  const long long units = (long long)p.batch * p.kv_heads;
  // chunks per group: as many as one wave of the GPU holds (two CTAs per SM), but chunks of
  // at most 4096 keys (partials stay small) and at least 256 keys (per-CTA setup stays
  // small).  Measured on few groups with long bands (64 groups of up to 16k keys): one wave
  // of 4 chunks per group beats two or more waves of shorter chunks.
  const long long slots = 2ll * sms;
  long long s = std::max<long long>(slots / units, (lmax + 4095) / 4096);
  s = std::min<long long>(s, std::max<long long>(1, (lmax + 255) / 256));
  s = std::min<long long>(s, kDecodeMaxSplits);
  d.splits = (int)std::max<long long>(1, s);
  // a launch that fits one wave (two CTAs on every SM) combines its chunks through
  // distributed shared memory; longer launches keep the workspace partials, since clusters
  // of up to 8 CTAs leave SMs of a GPC unused once CTAs queue for slots
  d.cluster = d.splits >= 2 && d.splits <= kDecodeMaxCluster && units * d.splits <= slots;
  return d;
}

WsLayout workspace_layout(const gqa_params &p, bool need_q_rot) {
  WsLayout w;
  const size_t es = p.dtype == GQA_F32 ? 4 : 2;
  size_t off = 0;
  if (need_q_rot) {
    w.q_rot_off = off;
    w.q_rot_bytes = (size_t)p.batch * p.q_len * p.q_heads * p.head_dim * es;
    off = align_up(off + w.q_rot_bytes, kAlign);
  }
  // the partials of the largest plan a GPU could choose (the splits grow with the SM count)
  DecodePlan d = decode_plan(p, kPlanMaxSms);
  if (d.eligible && d.splits > 1) {
    const size_t groups = (size_t)p.batch * p.kv_heads;
    const size_t slots = groups * d.splits;
    w.part_acc_off = off;
    w.part_acc_bytes = slots * d.rows * (p.v_head_dim ? p.v_head_dim : p.head_dim) * sizeof(float);
    off = align_up(off + w.part_acc_bytes, kAlign);
    w.part_ml_off = off;
    w.part_ml_bytes = slots * d.rows * 2 * sizeof(float);
    off = align_up(off + w.part_ml_bytes, kAlign);
    w.tickets_off = off;
    w.tickets_bytes = groups * sizeof(int32_t);
    off = align_up(off + w.tickets_bytes, kAlign);
  }
  // the block map of a boolean mask on the tensor-core prefill (any call with more than one
  // query token that the prefill kernel can take): one bit per (b, q head, 128-row query
  // tile, 16-key chunk of the cache), the largest any mask shape needs
  const int dv = p.v_head_dim ? p.v_head_dim : p.head_dim;
  if (p.q_len > 1 && p.dtype != GQA_F32 && dv == p.head_dim && (p.head_dim == 64 || p.head_dim == 128)) {
    w.blockmap_off = off;
    w.blockmap_bytes = (size_t)p.batch * p.q_heads * ((p.q_len + 127) / 128) * ((p.cap_present + 511) / 512) * 4;
    off = align_up(off + w.blockmap_bytes, kAlign);
  }
  w.total = off;
  return w;
}

namespace {

enum Mode { kPrefill, kDecode };

// Validate the pointers and fill a Call.  Returns GQA_OK or the first error.
gqa_status make_call(Call &c, const gqa_params *p, const void *q, const void *k, const void *v, const void *past_k,
                     const void *past_v, const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                     const float *head_sink, void *out, void *present_k, void *present_v, int32_t *dev_status,
                     void *stream) {
  gqa_status s = check_params(p);
  if (s != GQA_OK) return s;
  c.p = *p;
  if (c.p.scale == 0.f) c.p.scale = 1.f / sqrtf((float)p->head_dim);
  c.G = p->q_heads / p->kv_heads;
  c.Dv = p->v_head_dim ? p->v_head_dim : p->head_dim;
  c.esize = p->dtype == GQA_F32 ? 4 : 2;
  if (!q || !seqlens_k || !present_k || !present_v) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(present_k) || !aligned16(present_v)) return GQA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqlens_k) & 3u) || (reinterpret_cast<uintptr_t>(head_sink) & 3u))
    return GQA_ERR_INVALID_ARG;
  if ((k == nullptr) != (v == nullptr)) return GQA_ERR_INVALID_ARG;
  c.append = k != nullptr;
  if (c.append) {
    if (!aligned16(k) || !aligned16(v)) return GQA_ERR_INVALID_ARG;
    if ((past_k == nullptr) != (past_v == nullptr)) return GQA_ERR_INVALID_ARG;
    const bool alias_k = past_k == nullptr || past_k == present_k;
    const bool alias_v = past_v == nullptr || past_v == present_v;
    if (alias_k != alias_v) return GQA_ERR_INVALID_ARG;
    c.past_separate = !alias_k;
    if (c.past_separate && p->kv_ring) return GQA_ERR_INVALID_ARG;  // a ring is updated in place
    if (c.past_separate) {
      if (!aligned16(past_k) || !aligned16(past_v)) return GQA_ERR_INVALID_ARG;
      if (p->cap_past < 1) return GQA_ERR_CAPACITY;
    }
    if (p->do_rotary) {
      if (!cos_cache || !sin_cache || !aligned16(cos_cache) || !aligned16(sin_cache)) return GQA_ERR_INVALID_ARG;
    }
  } else {
    if (p->do_rotary) return GQA_ERR_INVALID_ARG;  // attention only: q arrives rotated
    c.past_separate = 0;
  }
  c.q_in = q;
  c.q = q;
  c.k = k;
  c.v = v;
  c.past_k = past_k;
  c.past_v = past_v;
  c.seqlens = seqlens_k;
  c.cos = cos_cache;
  c.sin = sin_cache;
  c.head_sink = head_sink;
  c.out = out;
  c.present_k = present_k;
  c.present_v = present_v;
  c.status = dev_status;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.wait_limit = g_test_stall.load(std::memory_order_relaxed);
  c.stall = c.wait_limit > 0;
  return GQA_OK;
}

// The tensor-core prefill reads the mask by TMA: 16-byte aligned data and strides.  Other
// masks go to the CUDA-core kernel.
bool mask_tma_ok(const Call &c) {
  const long long es = c.mask_kind == GQA_MASK_ADD ? 2 : 1;
  const long long lim = 1ll << 39;
  return (reinterpret_cast<uintptr_t>(c.mask) & 15u) == 0 && (c.mask_si * es) % 16 == 0 &&
         (c.mask_sh * es) % 16 == 0 && (c.mask_sb * es) % 16 == 0 && c.mask_si * es < lim && c.mask_sh * es < lim &&
         c.mask_sb * es < lim && (c.p.head_dim == 128 || c.p.head_dim == 64) && c.Dv == c.p.head_dim;
}

gqa_status run_attention(Mode mode, const gqa_params *p, const void *q, const void *k, const void *v,
                         const void *past_k, const void *past_v, const int32_t *seqlens_k, const void *cos_cache,
                         const void *sin_cache, const float *head_sink, void *out, void *present_k, void *present_v,
                         void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream,
                         const gqa_mask *mask = nullptr, const int64_t *nonpad = nullptr) {
  Call c;
  gqa_status s = make_call(c, p, q, k, v, past_k, past_v, nonpad ? reinterpret_cast<const int32_t *>(nonpad) : seqlens_k,
                           cos_cache, sin_cache, head_sink, out, present_k, present_v, dev_status, stream);
  if (s != GQA_OK) return s;
  if (nonpad) {  // a padded cache: the kernels read the valid lengths instead of seqlens_k
    c.seqlens = nullptr;
    c.nonpad = nonpad;
    if (mode == kPrefill && decode_plan(c.p, device_sm_count()).eligible) mode = kDecode;
  }
  if (!out || !aligned16(out)) return GQA_ERR_INVALID_ARG;
  const bool rotate = c.append && p->do_rotary;
  const WsLayout wl = workspace_layout(c.p, rotate);
  const DecodePlan dp = decode_plan(c.p, device_sm_count());
  // the split decode kernel appends and rotates itself; every other path runs K1 first
  const bool fused = mode == kDecode && dp.eligible;
  // a ring is read by the split decode kernel, and by the tensor-core prefill when its
  // 128-key tiles never straddle the wrap (capacity a multiple of 128; no mask)
  if (p->kv_ring && !fused &&
      (mode != kPrefill || p->dtype == GQA_F32 || mask || p->cap_present % 128 != 0))
    return GQA_ERR_UNSUPPORTED;
  if (mask) {
    if (!mask->data || (mask->kind != GQA_MASK_KEEP && mask->kind != GQA_MASK_ADD)) return GQA_ERR_INVALID_ARG;
    if (mask->kind == GQA_MASK_ADD && (reinterpret_cast<uintptr_t>(mask->data) & (c.esize - 1)))
      return GQA_ERR_INVALID_ARG;
    if (mask->keys < 1 || mask->stride_b < 0 || mask->stride_h < 0 || mask->stride_i < 0) return GQA_ERR_INVALID_ARG;
    c.mask = mask->data;
    c.mask_kind = mask->kind;
    c.mask_keys = mask->keys;
    c.mask_sb = mask->stride_b;
    c.mask_sh = mask->stride_h;
    c.mask_si = mask->stride_i;
  }
  size_t need = fused ? (dp.splits > 1 && !dp.cluster ? wl.total : 0) : (rotate ? wl.q_rot_off + wl.q_rot_bytes : 0);
  if (need > 0) {
    if (!workspace || !aligned16(workspace)) return GQA_ERR_WORKSPACE;
    if (workspace_bytes < need) return GQA_ERR_WORKSPACE;
  }
  c.ws = static_cast<char *>(workspace);
  c.ws_bytes = workspace_bytes;
  if (fused) {
    if (c.append && c.past_separate) {
      s = launch_copy_past(c);
      if (s != GQA_OK) return s;
    }
    return mask ? launch_decode_split_masked(c, dp, wl) : launch_decode_split(c, dp, wl);
  }
  if (c.append) {
    c.q_rot = rotate ? c.ws + wl.q_rot_off : nullptr;
    s = launch_rope_append(c);
    if (s != GQA_OK) return s;
    if (rotate) c.q = c.q_rot;
  }
  if (mode == kDecode || p->dtype == GQA_F32) return launch_attention_simt(c);
  if (mask) {
    if (!mask_tma_ok(c)) return launch_attention_simt(c);
    // a boolean mask's block map lets the prefill skip the key tiles it removes entirely,
    // when the workspace has room for it (it is optional)
    if (c.mask_kind == GQA_MASK_KEEP && wl.blockmap_bytes > 0 && c.ws && aligned16(c.ws) &&
        workspace_bytes >= wl.blockmap_off + wl.blockmap_bytes) {
      c.blockmap = reinterpret_cast<uint32_t *>(c.ws + wl.blockmap_off);
      c.blockmap_extent = wl.blockmap_bytes / 4;
    }
    return launch_prefill_tc_masked(c);
  }
  return launch_prefill_tc(c);
}

// Quantized cache (fmt 1: E4M3 codes, fmt 2: int8 codes): the step's K/V quantized on
// append, attention over code * scale.  The split decode kernel takes D = Dv = 128 shapes in
// its envelope; everything else runs the RoPE/append kernel and the CUDA-core kernel.
gqa_status run_attention_q8(Mode mode, int fmt, const gqa_params *p, const void *q, const void *k, const void *v,
                            const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                            const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                            uint8_t *present_k, uint8_t *present_v, void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, void *stream) {
  Call c;
  gqa_status s = make_call(c, p, q, k, v, nullptr, nullptr, seqlens_k, cos_cache, sin_cache, head_sink, out,
                           present_k, present_v, dev_status, stream);
  if (s != GQA_OK) return s;
  if (p->kv_ring) return GQA_ERR_UNSUPPORTED;
  if (!k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return GQA_ERR_INVALID_ARG;
  if (!out || !aligned16(out)) return GQA_ERR_INVALID_ARG;
  c.q8 = fmt;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  const bool rotate = c.append && p->do_rotary;
  const WsLayout wl = workspace_layout(c.p, rotate);
  const DecodePlan dp = decode_plan(c.p, device_sm_count());
  const bool fused = mode == kDecode && dp.eligible && p->head_dim == 128 && c.Dv == 128;
  const size_t need = fused ? (dp.splits > 1 && !dp.cluster ? wl.total : 0) : (rotate ? wl.q_rot_off + wl.q_rot_bytes : 0);
  if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need)) return GQA_ERR_WORKSPACE;
  c.ws = static_cast<char *>(workspace);
  c.ws_bytes = workspace_bytes;
  if (fused) return fmt == 2 ? launch_decode_split_i8(c, dp, wl) : launch_decode_split_q8(c, dp, wl);
  if (c.append) {
    c.q_rot = rotate ? c.ws + wl.q_rot_off : nullptr;
    s = launch_rope_append(c);
    if (s != GQA_OK) return s;
    if (rotate) c.q = c.q_rot;
  }
  return launch_attention_simt(c);
}

}  // namespace
}  // namespace gqa

extern "C" {

size_t gqa_workspace_bytes(const gqa_params *p) {
  if (gqa::check_params(p) != GQA_OK) return 0;
  return gqa::workspace_layout(*p, p->do_rotary != 0).total;
}

gqa_status gqa_attention_prefill(const gqa_params *p, const void *q, const void *k, const void *v,
                                 const void *past_k, const void *past_v, const int32_t *seqlens_k,
                                 const void *cos_cache, const void *sin_cache, const float *head_sink, void *out,
                                 void *present_k, void *present_v, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_attention(gqa::kPrefill, p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink,
                            out, present_k, present_v, workspace, workspace_bytes, dev_status, stream);
}

gqa_status gqa_attention_decode(const gqa_params *p, const void *q, const void *k, const void *v,
                                const void *past_k, const void *past_v, const int32_t *seqlens_k,
                                const void *cos_cache, const void *sin_cache, const float *head_sink, void *out,
                                void *present_k, void *present_v, void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_attention(gqa::kDecode, p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink,
                            out, present_k, present_v, workspace, workspace_bytes, dev_status, stream);
}

gqa_status gqa_attention_nonpad(const gqa_params *p, const int64_t *nonpad_kv_seqlen, const void *q,
                                const void *k_cache, const void *v_cache, const float *head_sink, void *out,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  if (!p || !nonpad_kv_seqlen || (reinterpret_cast<uintptr_t>(nonpad_kv_seqlen) & 7u)) return GQA_ERR_INVALID_ARG;
  if (p->kv_ring || p->do_rotary) return GQA_ERR_INVALID_ARG;  // a plain cache, q as given
  return gqa::run_attention(gqa::kPrefill, p, q, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                            head_sink, out, const_cast<void *>(k_cache), const_cast<void *>(v_cache), workspace,
                            workspace_bytes, dev_status, stream, nullptr, nonpad_kv_seqlen);
}

gqa_status gqa_attention_decode_masked(const gqa_params *p, const gqa_mask *mask, const void *q, const void *k,
                                       const void *v, const void *past_k, const void *past_v,
                                       const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                       const float *head_sink, void *out, void *present_k, void *present_v,
                                       void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                       void *stream) {
  GQA_TRACE_CALL();
  if (!mask) return GQA_ERR_INVALID_ARG;
  return gqa::run_attention(gqa::kDecode, p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink,
                            out, present_k, present_v, workspace, workspace_bytes, dev_status, stream, mask);
}

gqa_status gqa_attention_prefill_masked(const gqa_params *p, const gqa_mask *mask, const void *q, const void *k,
                                        const void *v, const void *past_k, const void *past_v,
                                        const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                        const float *head_sink, void *out, void *present_k, void *present_v,
                                        void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                        void *stream) {
  GQA_TRACE_CALL();
  if (!mask) return GQA_ERR_INVALID_ARG;
  return gqa::run_attention(gqa::kPrefill, p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink,
                            out, present_k, present_v, workspace, workspace_bytes, dev_status, stream, mask);
}

gqa_status gqa_attention_decode_q8(const gqa_params *p, const void *q, const void *k, const void *v,
                                   const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                   const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                   uint8_t *present_k, uint8_t *present_v, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_attention_q8(gqa::kDecode, 1, p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale,
                               v_scale, out, present_k, present_v, workspace, workspace_bytes, dev_status, stream);
}

gqa_status gqa_attention_prefill_q8(const gqa_params *p, const void *q, const void *k, const void *v,
                                    const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                    const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                    uint8_t *present_k, uint8_t *present_v, void *workspace, size_t workspace_bytes,
                                    int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_attention_q8(gqa::kPrefill, 1, p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale,
                               v_scale, out, present_k, present_v, workspace, workspace_bytes, dev_status, stream);
}

gqa_status gqa_attention_decode_i8(const gqa_params *p, const void *q, const void *k, const void *v,
                                   const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                   const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                   int8_t *present_k, int8_t *present_v, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_attention_q8(gqa::kDecode, 2, p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale,
                               v_scale, out, reinterpret_cast<uint8_t *>(present_k),
                               reinterpret_cast<uint8_t *>(present_v), workspace, workspace_bytes, dev_status, stream);
}

gqa_status gqa_attention_prefill_i8(const gqa_params *p, const void *q, const void *k, const void *v,
                                    const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                    const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                    int8_t *present_k, int8_t *present_v, void *workspace, size_t workspace_bytes,
                                    int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_attention_q8(gqa::kPrefill, 2, p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale,
                               v_scale, out, reinterpret_cast<uint8_t *>(present_k),
                               reinterpret_cast<uint8_t *>(present_v), workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"

namespace gqa {
namespace {

// A paged cache: decode runs the split-KV kernel (which appends through the table itself);
// prefill runs the RoPE/append kernel through the table, then the tensor-core prefill.
gqa_status run_paged(Mode mode, const gqa_params *p, const void *q, const void *k, const void *v,
                     const int32_t *seqlens_k, const int32_t *block_table, int32_t max_pages, int32_t num_pages,
                     const void *cos_cache, const void *sin_cache, const float *head_sink, void *out, void *k_pool,
                     void *v_pool, void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream) {
  Call c;
  gqa_status s = make_call(c, p, q, k, v, nullptr, nullptr, seqlens_k, cos_cache, sin_cache, head_sink, out, k_pool,
                           v_pool, dev_status, stream);
  if (s != GQA_OK) return s;
  if (p->kv_ring) return GQA_ERR_INVALID_ARG;
  if (c.Dv != p->head_dim) return GQA_ERR_UNSUPPORTED;  // pages hold K and V rows of one width
  if (!block_table || (reinterpret_cast<uintptr_t>(block_table) & 3u)) return GQA_ERR_INVALID_ARG;
  if (max_pages < 1 || num_pages < 1) return GQA_ERR_INVALID_ARG;
  if ((long long)max_pages * 64 != p->cap_present) return GQA_ERR_CAPACITY;
  if ((long long)num_pages * p->kv_heads > (1ll << 30)) return GQA_ERR_UNSUPPORTED;
  if (!out || !aligned16(out)) return GQA_ERR_INVALID_ARG;
  c.block_table = block_table;
  c.max_pages = max_pages;
  c.num_pages = num_pages;
  const bool rotate = c.append && p->do_rotary;
  const WsLayout wl = workspace_layout(c.p, rotate);
  if (mode == kDecode) {
    const DecodePlan dp = decode_plan(c.p, device_sm_count());
    if (!dp.eligible) return GQA_ERR_UNSUPPORTED;  // only the split decode kernel reads pages in decode
    const size_t need = dp.splits > 1 && !dp.cluster ? wl.total : 0;
    if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need)) return GQA_ERR_WORKSPACE;
    c.ws = static_cast<char *>(workspace);
    c.ws_bytes = workspace_bytes;
    return launch_decode_split(c, dp, wl);
  }
  if (p->dtype == GQA_F32) return GQA_ERR_UNSUPPORTED;  // the tensor-core prefill reads pages
  const size_t need = rotate ? wl.q_rot_off + wl.q_rot_bytes : 0;
  if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need)) return GQA_ERR_WORKSPACE;
  c.ws = static_cast<char *>(workspace);
  c.ws_bytes = workspace_bytes;
  if (c.append) {
    c.q_rot = rotate ? c.ws + wl.q_rot_off : nullptr;
    s = launch_rope_append(c);
    if (s != GQA_OK) return s;
    if (rotate) c.q = c.q_rot;
  }
  return launch_prefill_tc(c);
}

}  // namespace
}  // namespace gqa

extern "C" {

gqa_status gqa_attention_decode_paged(const gqa_params *p, const void *q, const void *k, const void *v,
                                      const int32_t *seqlens_k, const int32_t *block_table, int32_t max_pages,
                                      int32_t num_pages, const void *cos_cache, const void *sin_cache,
                                      const float *head_sink, void *out, void *k_pool, void *v_pool,
                                      void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                      void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_paged(gqa::kDecode, p, q, k, v, seqlens_k, block_table, max_pages, num_pages, cos_cache, sin_cache,
                        head_sink, out, k_pool, v_pool, workspace, workspace_bytes, dev_status, stream);
}

gqa_status gqa_attention_prefill_paged(const gqa_params *p, const void *q, const void *k, const void *v,
                                       const int32_t *seqlens_k, const int32_t *block_table, int32_t max_pages,
                                       int32_t num_pages, const void *cos_cache, const void *sin_cache,
                                       const float *head_sink, void *out, void *k_pool, void *v_pool,
                                       void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                       void *stream) {
  GQA_TRACE_CALL();
  return gqa::run_paged(gqa::kPrefill, p, q, k, v, seqlens_k, block_table, max_pages, num_pages, cos_cache,
                        sin_cache, head_sink, out, k_pool, v_pool, workspace, workspace_bytes, dev_status, stream);
}

gqa_status gqa_rope_append_kv(const gqa_params *p, const void *q, const void *k, const void *v, const void *past_k,
                              const void *past_v, const int32_t *seqlens_k, const void *cos_cache,
                              const void *sin_cache, void *q_rot, void *present_k, void *present_v,
                              int32_t *dev_status, void *stream) {
  GQA_TRACE_CALL();
  gqa::Call c;
  if (!k || !v) return GQA_ERR_INVALID_ARG;
  gqa_status s = gqa::make_call(c, p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, nullptr, nullptr,
                                present_k, present_v, dev_status, stream);
  if (s != GQA_OK) return s;
  if (q_rot && !gqa::aligned16(q_rot)) return GQA_ERR_INVALID_ARG;
  c.q_rot = q_rot;
  return gqa::launch_rope_append(c);
}

const char *gqa_status_string(gqa_status s) {
  switch (s) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument (shape, attribute, NULL or misaligned pointer)";
    case GQA_ERR_UNSUPPORTED: return "combination not supported by these kernels";
    case GQA_ERR_CAPACITY: return "capacity too small for the step";
    case GQA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case GQA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

int32_t gqa_abi_version(void) { return GQA_ABI_VERSION; }

#ifdef GQA_BOUNDS_CHECK
}  // extern "C"
namespace gqa {
namespace {
// one store inside a declared extent of 32 elements, one past it (the buffer itself is
// larger, so nothing leaves the allocation whether or not the guard works)
__global__ void bounds_probe_kernel(int32_t *buf, int32_t *status) {
  GQA_GUARD(8, 1, 32, status)
  buf[8] = 5;
  GQA_GUARD(40, 1, 32, status)
  buf[40] = 7;
}
}  // namespace
}  // namespace gqa
extern "C" {
/* Bounds-checked debug build only: checks that a guarded store outside its declared extent
 * is skipped and reported (buf: device int32 [64]). */
gqa_status gqa_test_bounds_check(int32_t *buf, int32_t *dev_status, void *stream) {
  if (!buf || !dev_status) return GQA_ERR_INVALID_ARG;
  gqa::bounds_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(buf, dev_status);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
#endif

gqa_status gqa_test_stall_waits(int64_t cycles) {
  if (cycles < 0) return GQA_ERR_INVALID_ARG;
  gqa::g_test_stall.store(cycles, std::memory_order_relaxed);
  return GQA_OK;
}

}  // extern "C"

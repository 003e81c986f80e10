// attn_simt.cu -- K5: attention on the CUDA cores in fp32, for fp32 inputs (where the
// tensor cores' TF32 cannot meet a 2e-5 error bound) and for decode shapes outside the
// split kernel's envelope (more than 32 query rows per kv head at D = 128).
//
// onnx-light-cpu "Attention Kernel Design", "Compute paths": the streaming recurrence
// keeps a running maximum, denominator and unnormalized output per query row while it
// visits key blocks; frontiers skip blocks that no row of the block can see.
// OpenVINO PR #37423, "Sliding window": a key is masked when q_abs - k_abs >= window.
// onnx-light-cpu "Layouts and semantics": an optional boolean mask removes keys like the
// band; an optional additive mask joins the scaled score before the softcap.
// The sink logit (PR #37423, "smooth_softmax / head_sink") joins the denominator at the
// end; a row with no visible key gives zeros ("Scheduling, precision, and invariants").
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace gqa {
namespace {

constexpr int kRows = 16;   // query rows per CTA (4 per warp)
constexpr int kKeys = 32;   // keys per shared-memory tile

struct SimtArgs {
  const void *q, *kc, *vc;  // q [B, curr, Hq, D]; caches [B, Hkv, cap, D] and [B, Hkv, cap, Dv]
  void *out;
  const int32_t *seqlens;
  const int64_t *nonpad;  // padded cache: valid keys per sequence (replaces seqlens)
  const float *head_sink;
  int32_t *status;
  int Hq, Hkv, G, D, Dv, curr, cap, cap_past, past_separate, rope_len, do_rotary, window, causal, has_sink;
  float scale, softcap;
  // attention mask (kind 0: none, 1: uint8 keep flags, 2: additive values of T), element
  // [b][hq][i][key] at b*msb + hq*msh + i*msi + key
  const void *mask;
  int mask_kind, mask_keys;
  long long msb, msh, msi;
  const float *k_scale, *v_scale;  // quantized cache: one scale per kv head (Q8 kernels)
  GQA_EXTENTS
};

// MASKED: a mask is given (compiled out otherwise); SAMEV: Dv == D (the common case keeps
// one load per element of both tiles and no V-width arithmetic); Q8: the caches hold
// one-byte codes (E4M3, or int8 when I8), the K scale joins the score scale and the V scale
// the output
template <typename T, bool MASKED, bool SAMEV, bool Q8, bool I8 = false>
__global__ void __launch_bounds__(128) attn_simt_kernel(SimtArgs a) {
  extern __shared__ float sm[];
  const int D = a.D, Dv = SAMEV ? a.D : a.Dv, Dw = SAMEV ? D : (D > Dv ? D : Dv);
  float *qs = sm;                          // [kRows][D]
  float *ks = qs + kRows * D;              // [kKeys][D + 1]
  float *vs = ks + kKeys * (D + 1);        // [kKeys][Dv]
  float *ps = vs + kKeys * Dv;             // [4 warps][kKeys]
  const int b = blockIdx.z, hq = blockIdx.y;
  const int i0 = blockIdx.x * kRows;
  const int hk = hq / a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int past = load_past(a.seqlens, a.nonpad, b, a.curr, a.cap);
  int st = sequence_status(past, a.curr, a.cap, a.cap_past, a.past_separate, a.do_rotary, a.rope_len);
  if (MASKED && !st && (long long)past + a.curr > a.mask_keys) st = GQA_DEV_BAD_SEQLEN;  // mask too short
  T *out = reinterpret_cast<T *>(a.out);
  const int nrows = min(kRows, a.curr - i0);
  if (st) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && hq == 0) report(a.status, st);
    for (int idx = threadIdx.x; idx < nrows * Dv; idx += blockDim.x) {
      int r = idx / Dv, d = idx % Dv;
      GQA_GUARD((((size_t)b * a.curr + i0 + r) * a.Hq + hq) * Dv + d, 1, a.ext.out, a.status)
      out[(((size_t)b * a.curr + i0 + r) * a.Hq + hq) * Dv + d] = from_f32<T>(0.f);
    }
    return;
  }
  const int total = past + a.curr;
  const T *q = reinterpret_cast<const T *>(a.q);
  for (int idx = threadIdx.x; idx < kRows * D; idx += blockDim.x) {
    int r = idx / D, d = idx % D;
    qs[idx] = r < nrows ? to_f32(q[(((size_t)b * a.curr + i0 + r) * a.Hq + hq) * D + d]) : 0.f;
  }
  // key frontier: the union of the rows' bands
  const int qa_lo = past + i0, qa_hi = past + i0 + nrows - 1;
  const int lo = a.window > 0 ? max(0, qa_lo - a.window + 1) : 0;
  const int hi = a.causal ? min(total, qa_hi + 1) : total;
  const T *kc = reinterpret_cast<const T *>(a.kc) + ((size_t)b * a.Hkv + hk) * a.cap * D;
  const T *vc = reinterpret_cast<const T *>(a.vc) + ((size_t)b * a.Hkv + hk) * a.cap * Dv;
  const uint8_t *kc8 = reinterpret_cast<const uint8_t *>(a.kc) + ((size_t)b * a.Hkv + hk) * a.cap * D;
  const uint8_t *vc8 = reinterpret_cast<const uint8_t *>(a.vc) + ((size_t)b * a.Hkv + hk) * a.cap * Dv;
  const float score_scale = Q8 ? a.scale * a.k_scale[hk] : a.scale;
  const float out_scale = Q8 ? a.v_scale[hk] : 1.f;
  constexpr int kMaxDSlots = 4;  // Dv <= 128
  float m[4], l[4], acc[4][kMaxDSlots];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    m[t] = -INFINITY;
    l[t] = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxDSlots; ++s) acc[t][s] = 0.f;
  }
  const int dslots = Dv / 32;
  for (int kt = lo; kt < hi; kt += kKeys) {
    __syncthreads();
    // one pass over both tiles, so the K and V loads of a thread are in flight together
    for (int idx = threadIdx.x; idx < kKeys * Dw; idx += blockDim.x) {
      const int j = idx / Dw, d = idx % Dw;
      const bool in = kt + j < hi;
      if (Q8) {
        if (SAMEV || d < D) ks[j * (D + 1) + d] = in ? code_to_f32<I8>(kc8[(size_t)(kt + j) * D + d]) : 0.f;
        if (SAMEV || d < Dv) vs[j * Dv + d] = in ? code_to_f32<I8>(vc8[(size_t)(kt + j) * Dv + d]) : 0.f;
      } else {
        if (SAMEV || d < D) ks[j * (D + 1) + d] = in ? to_f32(kc[(size_t)(kt + j) * D + d]) : 0.f;
        if (SAMEV || d < Dv) vs[j * Dv + d] = in ? to_f32(vc[(size_t)(kt + j) * Dv + d]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int r = warp * 4 + t;
      if (r >= nrows) break;
      const int qa = past + i0 + r;
      const int j = kt + lane;
      bool vis = j < hi && (!a.causal || j <= qa) && (a.window < 0 || qa - j < a.window);
      float bias = 0.f;
      if (MASKED && vis) {
        const long long mi = b * a.msb + hq * a.msh + (long long)(i0 + r) * a.msi + j;
        if (a.mask_kind == 1)
          vis = reinterpret_cast<const uint8_t *>(a.mask)[mi] != 0;
        else
          bias = to_f32(reinterpret_cast<const T *>(a.mask)[mi]);  // -inf: weight 0
      }
      float s = -INFINITY;
      if (vis) {
        float dot = 0.f;
        for (int d = 0; d < D; ++d) dot = fmaf(qs[r * D + d], ks[lane * (D + 1) + d], dot);
        s = dot * score_scale;
        if (MASKED && a.mask_kind == 2) s += bias;
        if (a.softcap > 0.f) s = a.softcap * tanhf(s / a.softcap);
      }
      float tmax = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_new = fmaxf(m[t], tmax);
      if (m_new == -INFINITY) continue;  // nothing visible to this row yet
      const float alpha = expf(m[t] - m_new);
      const float p = vis ? expf(s - m_new) : 0.f;
      float psum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[t] = l[t] * alpha + psum;
      m[t] = m_new;
      ps[warp * kKeys + lane] = p;
      __syncwarp();
#pragma unroll
      for (int s2 = 0; s2 < kMaxDSlots; ++s2) {
        if (s2 >= dslots) break;
        const int d = lane + 32 * s2;
        float x = acc[t][s2] * alpha;
        for (int jj = 0; jj < kKeys; ++jj) x = fmaf(ps[warp * kKeys + jj], vs[jj * Dv + d], x);
        acc[t][s2] = x;
      }
      __syncwarp();
    }
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int r = warp * 4 + t;
    if (r >= nrows) break;
    float num_scale = 1.f, den = l[t];
    if (m[t] == -INFINITY) {
      num_scale = 0.f;
      den = 1.f;  // no visible key: zeros with or without a sink
    } else if (a.has_sink) {
      const float z = a.head_sink ? a.head_sink[hq] : 0.f;
      const float mm = fmaxf(m[t], z);
      num_scale = expf(m[t] - mm);
      den = l[t] * num_scale + expf(z - mm);
    }
    for (int s2 = 0; s2 < dslots; ++s2) {
      const int d = lane + 32 * s2;
      GQA_GUARD((((size_t)b * a.curr + i0 + r) * a.Hq + hq) * Dv + d, 1, a.ext.out, a.status)
      out[(((size_t)b * a.curr + i0 + r) * a.Hq + hq) * Dv + d] = from_f32<T>(acc[t][s2] * num_scale / den * out_scale);
    }
  }
}

template <typename T> gqa_status launch_t(const Call &c) {
  const gqa_params &p = c.p;
  SimtArgs a;
  a.q = c.q;
  a.kc = c.present_k;
  a.vc = c.present_v;
  a.out = c.out;
  a.seqlens = c.seqlens;
  a.nonpad = c.nonpad;
  a.head_sink = c.head_sink;
  a.status = c.status;
  a.Hq = p.q_heads;
  a.Hkv = p.kv_heads;
  a.G = c.G;
  a.D = p.head_dim;
  a.Dv = c.Dv;
  a.curr = p.q_len;
  a.cap = p.cap_present;
  a.cap_past = p.cap_past;
  a.past_separate = c.past_separate;
  a.rope_len = p.rope_len;
  a.do_rotary = c.append ? p.do_rotary : 0;
  a.window = p.window;
  a.causal = p.causal;
  a.has_sink = (c.head_sink != nullptr) || p.smooth_softmax;
  a.scale = p.scale;
  a.softcap = p.softcap;
  a.mask = c.mask;
  a.mask_kind = c.mask ? c.mask_kind : 0;
  a.mask_keys = c.mask_keys;
  a.msb = c.mask_sb;
  a.msh = c.mask_sh;
  a.msi = c.mask_si;
  a.k_scale = c.k_scale;
  a.v_scale = c.v_scale;
#ifdef GQA_BOUNDS_CHECK
  a.ext = extents_of(c, WsLayout{});
#endif
  const int D = p.head_dim;
  size_t smem = sizeof(float) * (kRows * D + kKeys * (D + 1) + kKeys * c.Dv + 4 * kKeys);
  // D, Dv <= 128: at most 41.5 KB of shared memory, under the 48 KB default limit
  dim3 grid((p.q_len + kRows - 1) / kRows, p.q_heads, p.batch);
  const bool masked = c.mask != nullptr, samev = c.Dv == D;
  if (masked && c.q8) return GQA_ERR_UNSUPPORTED;
  auto kern = c.q8 == 2 ? (samev ? attn_simt_kernel<T, false, true, true, true> : attn_simt_kernel<T, false, false, true, true>)
              : c.q8 ? (samev ? attn_simt_kernel<T, false, true, true> : attn_simt_kernel<T, false, false, true>)
              : masked ? (samev ? attn_simt_kernel<T, true, true, false> : attn_simt_kernel<T, true, false, false>)
                       : (samev ? attn_simt_kernel<T, false, true, false> : attn_simt_kernel<T, false, false, false>);
  kern<<<grid, 128, smem, c.stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace

gqa_status launch_attention_simt(const Call &c) {
  switch (c.p.dtype) {
    case GQA_F32: return launch_t<float>(c);
    case GQA_F16: return launch_t<__half>(c);
    case GQA_BF16: return launch_t<__nv_bfloat16>(c);
  }
  return GQA_ERR_INVALID_ARG;
}

}  // namespace gqa

// rope_append.cu -- K1: RoPE (optional) + append of the step's keys/values into present,
// rotation of the queries, and the past -> present copy when the buffers are separate.
//
// tract PR #2645 "onnx: import GroupQueryAttention decode steps and its internal rotary",
// "What changed": past_key/past_value are concatenated with the step into present; with
// do_rotary the cos/sin cache halves are widened to the head size, positions run from
// seqlens_k (0 for a first prompt), and K is rotated before it enters the cache.
//
// Rotation of the half-split pair (x1, x2) = (x[d], x[d + D/2]) at position pos:
//   y1 = x1*c - x2*s,  y2 = x2*c + x1*s,  c, s = cos/sin_cache[pos, d]
// every product and every sum rounded to fp32 on its own (no FMA contraction), then the
// result rounded to the dtype with ties to even.  present is therefore bit-exact.
#include <limits.h>

#include "common.cuh"
#include "launch.h"

namespace gqa {
namespace {

template <typename T> struct Vec {
  static constexpr int N = 16 / sizeof(T);  // elements per 16-byte access
};

template <typename T>
__device__ __forceinline__ void rotate_chunk(const T *x1p, const T *x2p, const T *cp, const T *sp, T *y1p, T *y2p) {
  constexpr int N = Vec<T>::N;
  uint4 ux1 = *reinterpret_cast<const uint4 *>(x1p);
  uint4 ux2 = *reinterpret_cast<const uint4 *>(x2p);
  uint4 uc = *reinterpret_cast<const uint4 *>(cp);
  uint4 us = *reinterpret_cast<const uint4 *>(sp);
  const T *x1 = reinterpret_cast<const T *>(&ux1);
  const T *x2 = reinterpret_cast<const T *>(&ux2);
  const T *c = reinterpret_cast<const T *>(&uc);
  const T *s = reinterpret_cast<const T *>(&us);
  uint4 uy1, uy2;
  T *y1 = reinterpret_cast<T *>(&uy1);
  T *y2 = reinterpret_cast<T *>(&uy2);
#pragma unroll
  for (int e = 0; e < N; ++e) {
    float a1 = to_f32(x1[e]), a2 = to_f32(x2[e]), fc = to_f32(c[e]), fs = to_f32(s[e]);
    y1[e] = from_f32<T>(__fsub_rn(__fmul_rn(a1, fc), __fmul_rn(a2, fs)));
    y2[e] = from_f32<T>(__fadd_rn(__fmul_rn(a2, fc), __fmul_rn(a1, fs)));
  }
  *reinterpret_cast<uint4 *>(y1p) = uy1;
  *reinterpret_cast<uint4 *>(y2p) = uy2;
}

struct RopeArgs {
  const void *q, *k, *v, *cos, *sin;
  void *q_rot, *present_k, *present_v;
  const int32_t *seqlens;
  int32_t *status;
  int B, Hq, Hkv, D, Dv, curr, cap_present, cap_past, rope_len, do_rotary, past_separate;
  int ring;  // present is a ring: position p in slot p % cap_present
  // paged cache: present_k/v are pools [num_pages][Hkv][64][D]; table [B][max_pages] names the
  // page of positions [64n, 64n + 64); the pages of the step's band must all exist
  const int32_t *table;
  int max_pages, num_pages, window;
  // quantized cache: present_k/v hold one-byte codes of x / scale (fp32 division), one scale
  // per kv head: E4M3 when q8 == 1, int8 when q8 == 2
  int q8;
  const float *k_scale, *v_scale;
  GQA_EXTENTS
};

// N consecutive codes of x[e] / scale, stored as one N-byte word
template <typename T, int N, bool I8> __device__ __forceinline__ void store_codes(uint8_t *dst, const T *x, float scale) {
  uint32_t w[N / 4];
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    w[j] = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) w[j] |= (uint32_t)f32_to_code<I8>(__fdiv_rn(to_f32(x[4 * j + e]), scale)) << (8 * e);
  }
  if constexpr (N == 8)
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
  else
    *reinterpret_cast<uint32_t *>(dst) = w[0];
}

// One block per (b, i).  Work items: (head, chunk) over Hq q heads (when q_rot is wanted)
// and Hkv k heads, each N elements of each half of the row; then (v head, chunk) over Hkv
// v heads, N elements of a row of Dv each.
template <typename T>
__global__ void __launch_bounds__(256) rope_append_kernel(RopeArgs a) {
  constexpr int N = Vec<T>::N;
  const int b = blockIdx.x / a.curr;
  const int i = blockIdx.x % a.curr;
  const int past = a.seqlens[b];
  int st = sequence_status(past, a.curr, a.ring ? INT_MAX : a.cap_present, a.cap_past, a.past_separate,
                           a.do_rotary, a.rope_len);
  if (a.table && !st) {
    // every page the step reads or writes must exist (the same decision in every block of
    // the sequence and in the attention kernel: nothing of a rejected sequence is written)
    const int total = past + a.curr, lo = a.window > 0 ? max(0, past - a.window + 1) : 0;
    const int32_t *trow = a.table + (size_t)b * a.max_pages;
    bool bad = false;
    for (int n = lo / 64 + (int)threadIdx.x; n * 64 < total; n += blockDim.x) bad |= trow[n] < 0 || trow[n] >= a.num_pages;
    if (__syncthreads_or(bad)) st = GQA_DEV_BAD_PAGE;
  }
  if (st) {
    if (threadIdx.x == 0 && i == 0) report(a.status, st);
    return;
  }
  const int pos = past + i;
  const int half = a.D / 2;
  const int per_head = half / N;
  const int nq = a.q_rot ? a.Hq : 0;
  const int items_qk = (nq + a.Hkv) * per_head, v_per_head = a.Dv / N;
  const int items = items_qk + a.Hkv * v_per_head;
  const T *cosr = reinterpret_cast<const T *>(a.cos) + (size_t)pos * half;
  const T *sinr = reinterpret_cast<const T *>(a.sin) + (size_t)pos * half;
  const size_t slot = a.ring ? pos % a.cap_present : pos;
  // row of kv head h for this position: (b, h, slot), or (page, h, pos % 64) of a pool
  auto cache_row = [&](int h) -> size_t {
    if (a.table) return ((size_t)a.table[(size_t)b * a.max_pages + pos / 64] * a.Hkv + h) * 64 + pos % 64;
    return ((size_t)b * a.Hkv + h) * a.cap_present + slot;
  };
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    if (it >= items_qk) {  // v: a plain copy of one 16-byte chunk (or its codes)
      const int h = (it - items_qk) / v_per_head, c = ((it - items_qk) % v_per_head) * N;
      const T *src = reinterpret_cast<const T *>(a.v) + (((size_t)b * a.curr + i) * a.Hkv + h) * a.Dv;
      const size_t row = cache_row(h);
      GQA_GUARD(row * a.Dv + c, N, a.ext.pv, a.status)
      if (a.q8) {
        const uint4 x = *reinterpret_cast<const uint4 *>(src + c);
        uint8_t *v8 = reinterpret_cast<uint8_t *>(a.present_v) + row * a.Dv + c;
        if (a.q8 == 2)
          store_codes<T, N, true>(v8, reinterpret_cast<const T *>(&x), a.v_scale[h]);
        else
          store_codes<T, N, false>(v8, reinterpret_cast<const T *>(&x), a.v_scale[h]);
        continue;
      }
      T *dst = reinterpret_cast<T *>(a.present_v) + row * a.Dv;
      GQA_GUARD(row * a.Dv + c, N, a.ext.pv, a.status)
      *reinterpret_cast<uint4 *>(dst + c) = *reinterpret_cast<const uint4 *>(src + c);
      continue;
    }
    int head = it / per_head;
    int c = (it % per_head) * N;
    const T *src;
    T *dst;
    bool rot = a.do_rotary;
    [[maybe_unused]] size_t dst_off, dst_ext;  // the store's buffer: first element, extent
    if (head < nq) {
      size_t off = (((size_t)b * a.curr + i) * a.Hq + head) * a.D;
      src = reinterpret_cast<const T *>(a.q) + off;
      dst = reinterpret_cast<T *>(a.q_rot) + off;
      dst_off = off;
      dst_ext = GQA_EXT(qrot);
    } else {
      const int h = head - nq;
      src = reinterpret_cast<const T *>(a.k) + (((size_t)b * a.curr + i) * a.Hkv + h) * a.D;
      const size_t row = cache_row(h);
      if (a.q8) {  // the row in the dtype as without quantization, then its codes
        uint4 y1, y2;
        T *p1 = reinterpret_cast<T *>(&y1), *p2 = reinterpret_cast<T *>(&y2);
        if (rot) {
          rotate_chunk<T>(src + c, src + half + c, cosr + c, sinr + c, p1, p2);
        } else {
          y1 = *reinterpret_cast<const uint4 *>(src + c);
          y2 = *reinterpret_cast<const uint4 *>(src + half + c);
        }
        uint8_t *k8 = reinterpret_cast<uint8_t *>(a.present_k) + row * a.D;
        GQA_GUARD(row * a.D + c, half + N, a.ext.pk, a.status)
        if (a.q8 == 2) {
          store_codes<T, N, true>(k8 + c, p1, a.k_scale[h]);
          store_codes<T, N, true>(k8 + half + c, p2, a.k_scale[h]);
        } else {
          store_codes<T, N, false>(k8 + c, p1, a.k_scale[h]);
          store_codes<T, N, false>(k8 + half + c, p2, a.k_scale[h]);
        }
        continue;
      }
      dst = reinterpret_cast<T *>(a.present_k) + row * a.D;
      dst_off = row * a.D;
      dst_ext = GQA_EXT(pk);
    }
    GQA_GUARD(dst_off + c, half + N, dst_ext, a.status)
    if (rot) {
      rotate_chunk<T>(src + c, src + half + c, cosr + c, sinr + c, dst + c, dst + half + c);
    } else {
      *reinterpret_cast<uint4 *>(dst + c) = *reinterpret_cast<const uint4 *>(src + c);
      *reinterpret_cast<uint4 *>(dst + half + c) = *reinterpret_cast<const uint4 *>(src + half + c);
    }
  }
}

}  // namespace

// Copy rows [0, past_b) of past into present when the buffers are separate.  grid
// (B*Hkv, y): the y blocks of one (b, kv head) stride over its 16-byte words, K and V both.
template <typename T>
__global__ void __launch_bounds__(256) copy_past_words_kernel(const uint4 *past_k, const uint4 *past_v, uint4 *pres_k,
                                                              uint4 *pres_v, const int32_t *seqlens, int Hkv,
                                                              int cap_past, int cap_present, int D, int Dv,
                                                              int curr, int rope_len, int do_rotary,
                                                              [[maybe_unused]] Extents ext,
                                                              [[maybe_unused]] int32_t *status) {
  constexpr int N = 16 / sizeof(T);
  const int bh = blockIdx.x;
  const int b = bh / Hkv;
  const int past = seqlens[b];
  if (sequence_status(past, curr, cap_present, cap_past, 1, do_rotary, rope_len)) return;
  const size_t kw = (size_t)D / N, vw = (size_t)Dv / N;  // 16-byte words per K / V row
  const size_t kwords = (size_t)past * kw, words = kwords + (size_t)past * vw;
  const uint4 *sk = past_k + (size_t)bh * cap_past * kw;
  const uint4 *sv = past_v + (size_t)bh * cap_past * vw;
  uint4 *dk = pres_k + (size_t)bh * cap_present * kw;
  uint4 *dv = pres_v + (size_t)bh * cap_present * vw;
  for (size_t w = (size_t)blockIdx.y * blockDim.x + threadIdx.x; w < words; w += (size_t)gridDim.y * blockDim.x) {
    if (w < kwords) {
      GQA_GUARD(((size_t)bh * cap_present * kw + w) * N, N, ext.pk, status)
      dk[w] = sk[w];
    } else {
      GQA_GUARD(((size_t)bh * cap_present * vw + w - kwords) * N, N, ext.pv, status)
      dv[w - kwords] = sv[w - kwords];
    }
  }
}

template <typename T> static gqa_status launch_copy_t(const Call &c) {
  const gqa_params &p = c.p;
  dim3 grid(p.batch * p.kv_heads, 16);
  copy_past_words_kernel<T><<<grid, 256, 0, c.stream>>>(
      reinterpret_cast<const uint4 *>(c.past_k), reinterpret_cast<const uint4 *>(c.past_v),
      reinterpret_cast<uint4 *>(c.present_k), reinterpret_cast<uint4 *>(c.present_v), c.seqlens, p.kv_heads,
      p.cap_past, p.cap_present, p.head_dim, c.Dv, p.q_len, p.rope_len, p.do_rotary, extents_of(c, WsLayout{}),
      c.status);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

template <typename T> static gqa_status launch_t(const Call &c) {
  const gqa_params &p = c.p;
  RopeArgs a;
  a.q = c.q_in;
  a.k = c.k;
  a.v = c.v;
  a.cos = c.cos;
  a.sin = c.sin;
  a.q_rot = c.q_rot;
  a.present_k = c.present_k;
  a.present_v = c.present_v;
  a.seqlens = c.seqlens;
  a.status = c.status;
  a.B = p.batch;
  a.Hq = p.q_heads;
  a.Hkv = p.kv_heads;
  a.D = p.head_dim;
  a.Dv = c.Dv;
  a.curr = p.q_len;
  a.cap_present = p.cap_present;
  a.ring = p.kv_ring;
  a.table = c.block_table;
  a.max_pages = c.max_pages;
  a.num_pages = c.num_pages;
  a.window = p.window;
  a.cap_past = p.cap_past;
  a.rope_len = p.rope_len;
  a.do_rotary = p.do_rotary;
  a.past_separate = c.past_separate;
  a.q8 = c.q8;
  a.k_scale = c.k_scale;
  a.v_scale = c.v_scale;
#ifdef GQA_BOUNDS_CHECK
  a.ext = extents_of(c, WsLayout{});
#endif
  if (c.past_separate) {
    const gqa_status st = launch_copy_t<T>(c);
    if (st != GQA_OK) return st;
  }
  constexpr int N = Vec<T>::N;
  int items = ((c.q_rot ? p.q_heads : 0) + p.kv_heads) * (p.head_dim / 2 / N) + p.kv_heads * (c.Dv / N);
  int threads = items >= 256 ? 256 : ((items + 31) / 32) * 32;
  rope_append_kernel<T><<<p.batch * p.q_len, threads, 0, c.stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

gqa_status launch_copy_past(const Call &c) {
  switch (c.p.dtype) {
    case GQA_F32: return launch_copy_t<float>(c);
    case GQA_F16: return launch_copy_t<__half>(c);
    case GQA_BF16: return launch_copy_t<__nv_bfloat16>(c);
  }
  return GQA_ERR_INVALID_ARG;
}

gqa_status launch_rope_append(const Call &c) {
  switch (c.p.dtype) {
    case GQA_F32: return launch_t<float>(c);
    case GQA_F16: return launch_t<__half>(c);
    case GQA_BF16: return launch_t<__nv_bfloat16>(c);
  }
  return GQA_ERR_INVALID_ARG;
}

}  // namespace gqa

// decode_split.cu -- K3 + K4: split-KV decode with the combine fused into the last CTA.
//
// onnx-light-cpu "Attention Kernel Design": group_size = q_heads / kv_heads maps q heads
// onto kv heads without repeating K or V ("Layouts and semantics"); the streaming
// recurrence keeps a running max, denominator and unnormalized output per row and skips
// blocks outside the frontiers ("Compute paths"); fp32 accumulation, output narrowed once,
// fully masked rows give zeros ("Scheduling, precision, and invariants").
// OpenVINO PR #37423: window in true absolute positions, multi-token decode ("Sliding
// window"); sink logit in the denominator only ("smooth_softmax / head_sink").
// tract PR #2645, "What changed": bottom-right band, a decode token sees the whole cache.
//
// Work decomposition (one GB300, HBM-bound): the visible band of one (b, kv head) is
// [lo, total) with lo = max(0, past - window + 1); it is cut into chunks of `chunk` keys.
// CTA (chunk, kv head, b) holds all R = G*curr query rows of the group, so every K/V byte
// of the band is read from HBM exactly once.  A producer warp streams 64-key K and V tiles
// with TMA (128B-swizzled, NST-stage mbarrier ring); four consumer warps each take 16
// keys of a tile: S = Q K^T and O += P V on mma.sync (m16n8k16, fp32 accumulate), online
// softmax in the exp2 domain in registers.  The CTA merges its warps in shared memory and
// writes a partial (m, l, acc); the last CTA of the group (atomic ticket, no spin) adds
// the sink once, normalizes and writes the output.  A group with one chunk finishes
// in place without touching the workspace.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace gqa {
namespace {

constexpr int KT = 64;         // keys per tile
constexpr int kConsumers = 4;  // consumer warps (16 keys of a tile each)
constexpr int kThreads = (kConsumers + 1) * 32;

struct DecodeArgs {
  const void *q;        // [B, curr, Hq, D] (already rotated)
  void *out;            // [B, curr, Hq, D]
  const int32_t *seqlens;
  const float *head_sink;
  float *part_acc;      // [B*Hkv][max_chunks][R][D]
  float *part_ml;       // [B*Hkv][max_chunks][R][2]
  int32_t *tickets;     // [B*Hkv]
  int32_t *status;
  int Hq, Hkv, G, curr, R, cap, cap_past, past_separate, rope_len, do_rotary;
  int window, causal, chunk, max_chunks, has_sink;
  float score_mul;  // scale*log2(e), or scale/softcap with softcap
  float cap_mul;    // softcap*log2(e), 0 without softcap
};

template <int D, int MT, int NST> struct Smem {
  static constexpr int kTileBytes = KT * D * 2;       // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQRows = MT * 16;
  static constexpr int kQBytes = kQRows * D * 2;
  static constexpr int kStagesOff = 0;
  static constexpr int kQOff = NST * kStageBytes;
  static constexpr int kBarOff = kQOff + kQBytes;           // full[NST], empty[NST]
  static constexpr int kRedOff = kBarOff + 2 * NST * 8;     // red_m[4][QROWS], red_l[4][QROWS]
  static constexpr int kRowOff = kRedOff + 2 * kConsumers * kQRows * 4;  // row M, L
  static constexpr int kFlagOff = kRowOff + 2 * kQRows * 4;
  static constexpr int kBytes = kFlagOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
  static_assert(kQRows * D * 4 <= NST * kStageBytes, "merge buffer must fit in the stages");
};

template <typename T, int D, int MT, int NST>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        DecodeArgs a) {
  using L = Smem<D, MT, NST>;
  using M = Mma16816<T>;
  constexpr int QROWS = L::kQRows;
  constexpr int DCH = D / 8;  // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = smem + L::kStagesOff;
  uint8_t *qs = smem + L::kQOff;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
  uint64_t *empty = full + NST;
  float *red_m = reinterpret_cast<float *>(smem + L::kRedOff);
  float *red_l = red_m + kConsumers * QROWS;
  float *row_m = reinterpret_cast<float *>(smem + L::kRowOff);
  float *row_l = row_m + QROWS;
  volatile int *flags = reinterpret_cast<volatile int *>(smem + L::kFlagOff);  // [0] abort, [1] last

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int past = a.seqlens[b];
  const int st = sequence_status(past, a.curr, a.cap, a.cap_past, a.past_separate, a.do_rotary, a.rope_len);
  const int R = a.R;
  T *out = reinterpret_cast<T *>(a.out);

  if (st) {  // rejected sequence: zeros, reported once per sequence
    if (split == 0) {
      if (threadIdx.x == 0 && hkv == 0) report(a.status, st);
      for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
        int r = idx / D, d = idx % D;
        int i = r / a.G, g = r % a.G;
        out[(((size_t)b * a.curr + i) * a.Hq + hkv * a.G + g) * D + d] = from_f32<T>(0.f);
      }
    }
    return;
  }
  const int total = past + a.curr;
  const int lo = a.window > 0 ? max(0, past - a.window + 1) : 0;
  const int nchunks = (total - lo + a.chunk - 1) / a.chunk;
  if (split >= nchunks) return;  // whole CTA idle (uniform)
  const int c0 = lo + split * a.chunk;
  const int c1 = min(total, c0 + a.chunk);
  const int ntiles = (c1 - c0 + KT - 1) / KT;
  const int bh = b * a.Hkv + hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % NST;
        if (t >= NST && !mbar_wait(&empty[s], ((t / NST) - 1) & 1, flags)) break;
        mbar_expect_tx(&full[s], L::kStageBytes);
        const int kv0 = c0 + t * KT;
        uint8_t *kdst = stages + s * L::kStageBytes;
        uint8_t *vdst = kdst + L::kTileBytes;
#pragma unroll
        for (int db = 0; db < D / 64; ++db) {
          tma_load_3d(kdst + db * (KT * 128), &tmk, db * 64, kv0, bh, &full[s]);
          tma_load_3d(vdst + db * (KT * 128), &tmv, db * 64, kv0, bh, &full[s]);
        }
        ++issued;
      }
      if (flags[0]) {
        // drain: every copy issued must land before the CTA may exit
        volatile int no_abort = 0;
        for (int t = max(0, issued - NST); t < issued; ++t) mbar_wait(&full[t % NST], (t / NST) & 1, &no_abort);
        report(a.status, GQA_DEV_TIMEOUT);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumer warps
  const int cw = warp;
  // Q rows r = i*G + g (token i, q head hkv*G + g), 128B-swizzled in 64-column blocks
  {
    const T *q = reinterpret_cast<const T *>(a.q);
    for (int idx = threadIdx.x; idx < QROWS * DCH; idx += kConsumers * 32) {
      const int r = idx / DCH, ch = idx % DCH;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int i = r / a.G, g = r % a.G;
        val = *reinterpret_cast<const uint4 *>(q + (((size_t)b * a.curr + i) * a.Hq + hkv * a.G + g) * D + ch * 8);
      }
      *reinterpret_cast<uint4 *>(qs + (ch >> 3) * (QROWS * 128) + sw128(r, ch & 7)) = val;
    }
  }
  named_bar_sync(1, kConsumers * 32);

  float m[MT][2], l[MT][2];
  float acc[MT][D / 8][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m[mt][h] = -INFINITY;
      l[mt][h] = 0.f;
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][dn][e] = 0.f;
  }
  const uint32_t qs_u32 = smem_u32(qs);
  const int q_abs_min = past, q_abs_max = past + a.curr - 1;
  bool aborted = false;
  int t_fail = ntiles;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % NST;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (t / NST) & 1, flags))) {
      aborted = true;
      t_fail = t;
      break;
    }
    const int kv0 = c0 + t * KT;
    const int kb = kv0 + 16 * cw;  // this warp's first key
    const uint32_t ks_u32 = smem_u32(stages + s * L::kStageBytes);
    const uint32_t vs_u32 = ks_u32 + L::kTileBytes;

    // ---- S = Q K^T over this warp's 16 keys
    float sacc[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t kb0, kb1, kb2, kb3;
      {
        const int krow = 16 * cw + ((lane >> 4) << 3) + (lane & 7);
        const int kch = 2 * ks + ((lane >> 3) & 1);
        ldsm_x4(ks_u32 + (kch >> 3) * (KT * 128) + sw128(krow, kch & 7), kb0, kb1, kb2, kb3);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t af[4];
        const int qrow = 16 * mt + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int qch = 2 * ks + (lane >> 4);
        ldsm_x4(qs_u32 + (qch >> 3) * (QROWS * 128) + sw128(qrow, qch & 7), af[0], af[1], af[2], af[3]);
        M::run(sacc[mt][0], af, kb0, kb1);
        M::run(sacc[mt][1], af, kb2, kb3);
      }
    }

    // ---- scale, softcap, band mask (only on tiles that cross a frontier)
    const bool edge = !(kb >= c0 && kb + 15 < c1 && (!a.causal || kb + 15 <= q_abs_min) &&
                        (a.window < 0 || q_abs_max - kb < a.window));
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = sacc[mt][n][e];
          x = a.cap_mul != 0.f ? tanh_fast(x * a.score_mul) * a.cap_mul : x * a.score_mul;
          if (edge) {
            const int row = 16 * mt + (lane >> 2) + ((e >> 1) << 3);
            const int key = kb + 8 * n + 2 * (lane & 3) + (e & 1);
            const int qa = past + row / a.G;
            const bool vis = row < R && key >= c0 && key < c1 && (!a.causal || key <= qa) &&
                             (a.window < 0 || qa - key < a.window);
            if (!vis) x = -INFINITY;
          }
          sacc[mt][n][e] = x;
        }

    // ---- online softmax (exp2 domain); rows lane/4 (h=0) and lane/4+8 (h=1)
    uint32_t pa[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      float p[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = fmaxf(fmaxf(sacc[mt][0][2 * h], sacc[mt][0][2 * h + 1]),
                         fmaxf(sacc[mt][1][2 * h], sacc[mt][1][2 * h + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m[mt][h], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2(m[mt][h] - m_use);
        m[mt][h] = m_new;
        float rs = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = ex2(sacc[mt][n][2 * h + e] - m_use);
            p[n][2 * h + e] = pv;
            rs += pv;
          }
        l[mt][h] = l[mt][h] * alpha + rs;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          acc[mt][dn][2 * h] *= alpha;
          acc[mt][dn][2 * h + 1] *= alpha;
        }
      }
      pa[mt][0] = M::pack(p[0][0], p[0][1]);
      pa[mt][1] = M::pack(p[0][2], p[0][3]);
      pa[mt][2] = M::pack(p[1][0], p[1][1]);
      pa[mt][3] = M::pack(p[1][2], p[1][3]);
    }

    // ---- stale V rows (slots >= total) may hold NaN/Inf: zero them so 0 * V stays 0
    const bool stale = kb + 16 > total;
    if (stale) {
      const int first = max(0, total - kb);
      for (int idx = lane; idx < (16 - first) * DCH; idx += 32) {
        const int r = 16 * cw + first + idx / DCH, ch = idx % DCH;
        *reinterpret_cast<uint4 *>(stages + s * L::kStageBytes + L::kTileBytes + (ch >> 3) * (KT * 128) +
                                   sw128(r, ch & 7)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    // ---- O += P V over this warp's 16 keys
#pragma unroll
    for (int dd = 0; dd < D / 16; ++dd) {
      uint32_t v0, v1, v2, v3;
      const int vrow = 16 * cw + ((lane >> 3) & 1) * 8 + (lane & 7);
      const int vch = 2 * dd + (lane >> 4);
      ldsm_x4_t(vs_u32 + (vch >> 3) * (KT * 128) + sw128(vrow, vch & 7), v0, v1, v2, v3);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        M::run(acc[mt][2 * dd], pa[mt], v0, v1);
        M::run(acc[mt][2 * dd + 1], pa[mt], v2, v3);
      }
    }
    if (stale) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // -------------------------------------------------------------- merge the 4 warps
  // one decision for all consumer warps: a timed-out wait anywhere aborts the whole CTA
  aborted = named_bar_or(1, kConsumers * 32, aborted || flags[0] != 0);
  if (aborted) {
    // a wait timed out: the producer drains its copies and reports; take part in the
    // ticket so the group's counter stays consistent, write nothing
    if (cw == 0 && lane == 0) {
      // copies the producer may still have in flight must land before the CTA exits
      volatile int no_abort = 0;
      for (int t = t_fail; t < min(ntiles, t_fail + NST); ++t) mbar_wait(&full[t % NST], (t / NST) & 1, &no_abort);
      report(a.status, GQA_DEV_TIMEOUT);
      if (nchunks > 1) {
        __threadfence();
        const int old = atomicAdd(&a.tickets[bh], 1);
        if (old == nchunks - 1) a.tickets[bh] = 0;
      }
    }
    return;
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float lv = l[mt][h];
      lv += __shfl_xor_sync(0xffffffffu, lv, 1);
      lv += __shfl_xor_sync(0xffffffffu, lv, 2);
      l[mt][h] = lv;
      if ((lane & 3) == 0) {
        const int row = 16 * mt + (lane >> 2) + 8 * h;
        red_m[cw * QROWS + row] = m[mt][h];
        red_l[cw * QROWS + row] = lv;
      }
    }
  float *accbuf = reinterpret_cast<float *>(stages);  // [QROWS][D], stages are free now
  named_bar_sync(1, kConsumers * 32);
  if (threadIdx.x < QROWS) {
    const int row = threadIdx.x;
    float mm = -INFINITY;
    for (int w = 0; w < kConsumers; ++w) mm = fmaxf(mm, red_m[w * QROWS + row]);
    const float mu = mm == -INFINITY ? 0.f : mm;
    float ll = 0.f;
    for (int w = 0; w < kConsumers; ++w) ll += red_l[w * QROWS + row] * ex2(red_m[w * QROWS + row] - mu);
    row_m[row] = mm;
    row_l[row] = ll;
  }
  named_bar_sync(1, kConsumers * 32);
  // warps add their rescaled accumulators one after another (fixed order: deterministic)
  for (int w = 0; w < kConsumers; ++w) {
    if (cw == w) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = 16 * mt + (lane >> 2) + 8 * h;
          const float mm = row_m[row];
          const float f = ex2(m[mt][h] - (mm == -INFINITY ? 0.f : mm));
#pragma unroll
          for (int dn = 0; dn < D / 8; ++dn) {
            float2 *dst = reinterpret_cast<float2 *>(&accbuf[row * D + 8 * dn + 2 * (lane & 3)]);
            float2 prev = w == 0 ? make_float2(0.f, 0.f) : *dst;
            *dst = make_float2(prev.x + acc[mt][dn][2 * h] * f, prev.y + acc[mt][dn][2 * h + 1] * f);
          }
        }
    }
    named_bar_sync(1, kConsumers * 32);
  }

  if (nchunks == 1) {
    // ------------------------------------------------------------ finish in place
    for (int idx = threadIdx.x; idx < R * D; idx += kConsumers * 32) {
      const int r = idx / D, d = idx % D;
      const int i = r / a.G, g = r % a.G, hq = hkv * a.G + g;
      const float mm = row_m[r];
      float num = 0.f, den = 1.f;
      if (mm != -INFINITY) {
        float top = mm, sink_term = 0.f;
        if (a.has_sink) {
          const float z = (a.head_sink ? a.head_sink[hq] : 0.f) * kLog2e;
          top = fmaxf(mm, z);
          sink_term = ex2(z - top);
        }
        const float f = ex2(mm - top);
        num = accbuf[idx] * f;
        den = row_l[r] * f + sink_term;
      }
      out[(((size_t)b * a.curr + i) * a.Hq + hq) * D + d] = from_f32<T>(num / den);
    }
    return;
  }

  // -------------------------------------------------------------- write the partial
  {
    const size_t base = ((size_t)bh * a.max_chunks + split) * R;
    float4 *pacc = reinterpret_cast<float4 *>(a.part_acc + base * D);
    const float4 *src = reinterpret_cast<const float4 *>(accbuf);
    for (int idx = threadIdx.x; idx < R * D / 4; idx += kConsumers * 32) pacc[idx] = src[idx];
    for (int r = threadIdx.x; r < R; r += kConsumers * 32) {
      a.part_ml[(base + r) * 2] = row_m[r];
      a.part_ml[(base + r) * 2 + 1] = row_l[r];
    }
  }
  __threadfence();
  named_bar_sync(1, kConsumers * 32);
  if (threadIdx.x == 0) {
    const int old = atomicAdd(&a.tickets[bh], 1);
    flags[1] = old == nchunks - 1;
  }
  named_bar_sync(1, kConsumers * 32);
  if (!flags[1]) return;

  // -------------------------------------------------------------- last CTA: combine
  __threadfence();
  if (threadIdx.x == 0) a.tickets[bh] = 0;
  const size_t gbase = (size_t)bh * a.max_chunks * R;
  // per row: M over chunks (and the sink), L = sum l_c 2^(m_c - M) + sink term
  for (int r = threadIdx.x; r < R; r += kConsumers * 32) {
    const int hq = hkv * a.G + r % a.G;
    float mm = -INFINITY;
    for (int c = 0; c < nchunks; ++c) mm = fmaxf(mm, __ldcg(&a.part_ml[(gbase + (size_t)c * R + r) * 2]));
    float top = mm, sink_term = 0.f;
    if (mm != -INFINITY && a.has_sink) {
      const float z = (a.head_sink ? a.head_sink[hq] : 0.f) * kLog2e;
      top = fmaxf(mm, z);
      sink_term = ex2(z - top);
    }
    float ll = sink_term;
    if (mm != -INFINITY)
      for (int c = 0; c < nchunks; ++c) {
        const float mc = __ldcg(&a.part_ml[(gbase + (size_t)c * R + r) * 2]);
        ll += __ldcg(&a.part_ml[(gbase + (size_t)c * R + r) * 2 + 1]) * ex2(mc - top);
      }
    row_m[r] = mm == -INFINITY ? -INFINITY : top;
    row_l[r] = ll;
  }
  named_bar_sync(1, kConsumers * 32);
  for (int idx = threadIdx.x; idx < R * (D / 4); idx += kConsumers * 32) {
    const int r = idx / (D / 4), d4 = idx % (D / 4);
    const int i = r / a.G, g = r % a.G, hq = hkv * a.G + g;
    const float top = row_m[r];
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 1.f;
    if (top != -INFINITY) {
      for (int c = 0; c < nchunks; ++c) {
        const float mc = __ldcg(&a.part_ml[(gbase + (size_t)c * R + r) * 2]);
        if (mc == -INFINITY) continue;
        const float f = ex2(mc - top);
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part_acc + (gbase + (size_t)c * R + r) * D) + d4);
        sum.x += v.x * f;
        sum.y += v.y * f;
        sum.z += v.z * f;
        sum.w += v.w * f;
      }
      den = row_l[r];
    }
    T *o = out + (((size_t)b * a.curr + i) * a.Hq + hq) * D + d4 * 4;
    o[0] = from_f32<T>(sum.x / den);
    o[1] = from_f32<T>(sum.y / den);
    o[2] = from_f32<T>(sum.z / den);
    o[3] = from_f32<T>(sum.w / den);
  }
}

template <typename T, int D, int MT, int NST>
gqa_status launch_cfg(const Call &c, const DecodePlan &dp, const WsLayout &wl, const DecodeArgs &a) {
  using L = Smem<D, MT, NST>;
  CUtensorMap tk, tv;
  const long long outer = (long long)c.p.batch * c.p.kv_heads;
  if (!encode_kv_map(&tk, c.present_k, D, c.p.cap_present, outer, KT, 2)) return GQA_ERR_CUDA;
  if (!encode_kv_map(&tv, c.present_v, D, c.p.cap_present, outer, KT, 2)) return GQA_ERR_CUDA;
  auto kern = decode_split_kernel<T, D, MT, NST>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess)
    return GQA_ERR_CUDA;
  dim3 grid(dp.max_chunks, c.p.kv_heads, c.p.batch);
  kern<<<grid, kThreads, L::kAlloc, c.stream>>>(tk, tv, a);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

template <typename T>
gqa_status launch_t(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  const gqa_params &p = c.p;
  DecodeArgs a;
  a.q = c.q;
  a.out = c.out;
  a.seqlens = c.seqlens;
  a.head_sink = c.head_sink;
  a.part_acc = reinterpret_cast<float *>(c.ws + wl.part_acc_off);
  a.part_ml = reinterpret_cast<float *>(c.ws + wl.part_ml_off);
  a.tickets = reinterpret_cast<int32_t *>(c.ws + wl.tickets_off);
  a.status = c.status;
  a.Hq = p.q_heads;
  a.Hkv = p.kv_heads;
  a.G = c.G;
  a.curr = p.q_len;
  a.R = dp.rows;
  a.cap = p.cap_present;
  a.cap_past = p.cap_past;
  a.past_separate = c.past_separate;
  a.rope_len = p.rope_len;
  a.do_rotary = c.append ? p.do_rotary : 0;
  a.window = p.window;
  a.causal = p.causal;
  a.chunk = dp.chunk;
  a.max_chunks = dp.max_chunks;
  a.has_sink = (c.head_sink != nullptr) || p.smooth_softmax;
  if (p.softcap > 0.f) {
    a.score_mul = p.scale / p.softcap;
    a.cap_mul = p.softcap * kLog2e;
  } else {
    a.score_mul = p.scale * kLog2e;
    a.cap_mul = 0.f;
  }
  if (p.head_dim == 128) {
    switch (dp.mtiles) {
      case 1: return launch_cfg<T, 128, 1, 3>(c, dp, wl, a);
      case 2: return launch_cfg<T, 128, 2, 3>(c, dp, wl, a);
    }
  } else if (p.head_dim == 64) {
    switch (dp.mtiles) {
      case 1: return launch_cfg<T, 64, 1, 6>(c, dp, wl, a);
      case 2: return launch_cfg<T, 64, 2, 6>(c, dp, wl, a);
      case 3: return launch_cfg<T, 64, 3, 6>(c, dp, wl, a);
      case 4: return launch_cfg<T, 64, 4, 6>(c, dp, wl, a);
    }
  }
  return GQA_ERR_UNSUPPORTED;
}

}  // namespace

gqa_status launch_decode_split(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  switch (c.p.dtype) {
    case GQA_F16: return launch_t<__half>(c, dp, wl);
    case GQA_BF16: return launch_t<__nv_bfloat16>(c, dp, wl);
  }
  return GQA_ERR_UNSUPPORTED;
}

}  // namespace gqa

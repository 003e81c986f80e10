#pragma once
#include <type_traits>
// decode_split.cuh -- K3 + K4: split-KV decode with RoPE + append fused in and the combine
// done by the last CTA of each (b, kv head) group.
//
// onnx-light-cpu "Attention Kernel Design": group_size = q_heads / kv_heads maps q heads
// onto kv heads without repeating K or V ("Layouts and semantics"); the streaming
// recurrence keeps a running max, denominator and unnormalized output per row and skips
// blocks outside the frontiers ("Compute paths"); fp32 accumulation, output narrowed once,
// fully masked rows give zeros ("Scheduling, precision, and invariants").
// OpenVINO PR #37423: window in true absolute positions, multi-token decode ("Sliding
// window"); sink logit in the denominator only ("smooth_softmax / head_sink").
// tract PR #2645, "What changed": the step's K (rotated) and V are appended to the cache at
// seqlens_k and the query is rotated at the same positions; bottom-right band.
//
// Work decomposition (one GB300, HBM-bound): the visible band of group (b, kv head) is
// [lo, total) with lo = max(0, past - window + 1); it is cut into S equal chunks (rounded
// up to 64-key tiles, so no tile is read twice), one CTA each: CTA (chunk, kv head, b)
// holds all R = G*curr query rows of the group and reads every K/V byte of its chunk once.
// Each group's chunks are equal, so long and short sequences balance within a group; two
// CTAs share an SM so one's prologue and epilogue overlap the other's streaming.
//
// Pipeline: four warps, each takes 16 keys of every 64-key tile: S = Q K^T and O += P V on
// mma.sync m16n8k16 (fp32 accumulate), online softmax in the exp2 domain with a lazily
// moved reference max.  A group of at most 8 query rows runs the transposed products
// S^T = K Q^T and O^T += V^T P^T instead (keys, then V's head dims, as the MMA's 16-row
// side; the rows as its 8 columns), which halves the MMAs.  K and V tiles arrive by TMA
// (128B swizzle) through an NST-stage mbarrier ring; the last of the four warps to release
// a stage refills it, and before loading the tile that holds the group's new rows it
// writes them to present (K rotated) so the TMA reads them back.  The CTA merges its warps in shared memory; a
// one-chunk group finishes in place, otherwise the CTA writes (m, l, acc) and the last CTA
// of the group (atomic ticket, no spin-wait) adds the sink once, normalizes and writes out.
// Launched with programmatic stream serialization: the prologue overlaps the previous
// kernel's tail and griddepcontrol.wait orders every global read after it.
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace gqa {
namespace {

constexpr int KT = 64;         // keys per tile
constexpr int kWarps = 4;      // 16 keys of a tile each
constexpr int kThreads = kWarps * 32;
constexpr float kRescaleLog2 = 8.f;  // move the reference max only when it grows by > 2^8
constexpr int kMaxSplits = kDecodeMaxSplits;
constexpr int kMaxCluster = kDecodeMaxCluster;  // chunks combined through distributed shared memory

struct DecodeArgs {
  const void *q;          // [B, curr, Hq, D] as given (rotated here when do_rotary)
  const void *k, *v;      // [B, curr, Hkv, D] / [B, curr, Hkv, DV] new rows, or NULL (attention only)
  const void *cos, *sin;  // [rope_len, D/2]
  void *present_k, *present_v;
  void *out;              // [B, curr, Hq, DV]
  const int32_t *seqlens;
  const int64_t *nonpad;  // padded cache: valid keys per sequence (replaces seqlens)
  const float *head_sink;
  float *part_acc;      // [B*Hkv][S][R][DV]
  float *part_ml;       // [B*Hkv][S][R][2]
  int32_t *tickets;     // [B*Hkv]
  int32_t *status;
  int Hq, Hkv, G, curr, R, cap, cap_past, past_separate, rope_len, do_rotary, append;
  int window, causal, splits, has_sink, ring;
  const int32_t *table;  // paged cache: [B][max_pages] page of positions [64n, 64n + 64); null otherwise
  int max_pages, num_pages;
  // attention mask (masked kernels only): element [b][hq][i][key] at
  // b*msb + hq*msh + i*msi + key; kind 1 = uint8 keep flags, 2 = additive values of T
  const void *mask;
  long long msb, msh, msi;
  int mask_kind, mask_keys;
  float mask_mul;  // 1 / scale: an additive value joins the raw dot product before scaling
  float score_mul;  // scale*log2(e), or scale/softcap with softcap
  float cap_mul;    // softcap*log2(e), 0 without softcap
  const float *k_scale, *v_scale;  // f8 cache (Q8 kernels): one scale per kv head
  long long wait_limit;  // SM cycles after which a pipeline wait gives up
  int stall;             // test hook: the first wait is on a barrier nothing completes
  GQA_EXTENTS
};

template <int D, int DV, int MT, int NST, bool Q8 = false> struct Smem {
  static constexpr int kEs = Q8 ? 1 : 2;  // bytes per cached element (E4M3 codes or the dtype)
  static constexpr int kTileBytes = KT * D * kEs;  // one K tile; the V tile follows it
  static constexpr int kVTileBytes = KT * DV * kEs;
  static constexpr int kStageBytes = kTileBytes + kVTileBytes;
  // Q8, 16-row form: every warp widens the V codes of its 16 keys of the stage to f16 here
  // (the layout of a 16-bit V tile), right after the stages, so the two form one region for
  // the merge below; K codes go from the stage straight into MMA fragments
  static constexpr int kConvBytes = Q8 ? KT * DV * 2 : 0;
  static constexpr int kReuseBytes = NST * kStageBytes + kConvBytes;
  static constexpr int kQRows = MT * 16;
  static constexpr int kStagesOff = 0;
  static constexpr int kConvOff = NST * kStageBytes;
  static constexpr int kQOff = kReuseBytes;
  static constexpr int kBarOff = kQOff + kQRows * D * 2;                  // full[NST], xbar, stall
  static constexpr int kRedOff = kBarOff + (NST + 2) * 8;                 // red_m, red_l [4][QROWS]
  static constexpr int kRowOff = kRedOff + 2 * kWarps * kQRows * 4;       // row_m, row_l, sink [QROWS]
  static constexpr int kFlagOff = kRowOff + 3 * kQRows * 4;
  // per stage: how many warps are done with its current tile (counts up, never reset);
  // then the number of tiles issued so far
  static constexpr int kCntOff = kFlagOff + 16;
  // the step's new K and V rows of this kv head, copied in at the start when they fit
  static constexpr int kNewOff = (kCntOff + (NST + 1) * 4 + 15) / 16 * 16;
  static constexpr int kNewBytes = 2048;
  // cluster combine: the partials the other chunks send to this CTA, in a region of their
  // own when they fit (one 16-row MMA tile), so that peers may send before this CTA has
  // finished streaming
  static constexpr int kRcvOff = kNewOff + kNewBytes;
  static constexpr int kRcvBytes = MT == 1 ? 5120 : 0;
  static constexpr int kBytes = kRcvOff + kRcvBytes;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
  // per-warp merge regions (rows padded by 4 floats: the fragment stores of one warp
  // instruction then spread over all banks) and the combine's chunk statistics reuse the stages
  static constexpr int kAccStride = DV + 4;
  static_assert(kWarps * kQRows * kAccStride * 4 <= kReuseBytes, "merge regions must fit in the stages");
  static_assert(2 * kMaxSplits * kQRows * 4 <= kReuseBytes, "chunk statistics must fit in the stages");
  static_assert((kWarps * kQRows * kAccStride + kQRows * DV + 4 * kMaxCluster + 2 * kMaxCluster * kQRows) * 4 <=
                    kReuseBytes,
                "cluster exchange buffers must fit in the stages");
};

// four consecutive outputs in one 8-byte store
template <typename T> __device__ __forceinline__ void store4(T *o, float x, float y, float z, float w) {
  union {
    T e[4];
    uint2 u;
  } v;
  v.e[0] = from_f32<T>(x);
  v.e[1] = from_f32<T>(y);
  v.e[2] = from_f32<T>(z);
  v.e[3] = from_f32<T>(w);
  *reinterpret_cast<uint2 *>(o) = v.u;
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <typename T>
__device__ __forceinline__ void rotate8(const T *x1p, const T *x2p, const T *cp, const T *sp, uint4 &o1, uint4 &o2) {
  uint4 ux1 = *reinterpret_cast<const uint4 *>(x1p), ux2 = *reinterpret_cast<const uint4 *>(x2p);
  uint4 uc = *reinterpret_cast<const uint4 *>(cp), us = *reinterpret_cast<const uint4 *>(sp);
  const T *x1 = reinterpret_cast<const T *>(&ux1), *x2 = reinterpret_cast<const T *>(&ux2);
  const T *c = reinterpret_cast<const T *>(&uc), *s = reinterpret_cast<const T *>(&us);
  T *y1 = reinterpret_cast<T *>(&o1), *y2 = reinterpret_cast<T *>(&o2);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float a1 = to_f32(x1[e]), a2 = to_f32(x2[e]), fc = to_f32(c[e]), fs = to_f32(s[e]);
    y1[e] = from_f32<T>(__fsub_rn(__fmul_rn(a1, fc), __fmul_rn(a2, fs)));
    y2[e] = from_f32<T>(__fadd_rn(__fmul_rn(a2, fc), __fmul_rn(a1, fs)));
  }
}

// Eight values of the dtype as eight codes (E4M3, or int8 when I8) of x / scale (fp32
// division), one 8-byte word.
template <typename T, bool I8> __device__ __forceinline__ uint2 codes8(const uint4 &x, float scale) {
  const T *e = reinterpret_cast<const T *>(&x);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j >> 2] |= (uint32_t)f32_to_code<I8>(__fdiv_rn(to_f32(e[j]), scale)) << (8 * (j & 3));
  return make_uint2(w[0], w[1]);
}

// Eight values of the dtype as eight f16 values (exact for any value in the f16 range).
template <typename T> __device__ __forceinline__ uint4 to_half8(const uint4 &x) {
  const T *e = reinterpret_cast<const T *>(&x);
  uint4 r;
  uint32_t *w = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 h = __floats2half2_rn(to_f32(e[2 * j]), to_f32(e[2 * j + 1]));
    w[j] = *reinterpret_cast<const uint32_t *>(&h);
  }
  return r;
}

// Sixteen E4M3 codes (one 16-byte chunk) as sixteen f16 values, two 16-byte chunks: one pair
// conversion per two neighbouring codes (the low byte of the pair becomes the low half, as
// the f16 pair layout of a 16-bit tile wants; the lane order was checked on the GPU).
template <bool I8> __device__ __forceinline__ void widen16(const uint4 &codes, uint4 &lo, uint4 &hi) {
  const uint32_t in[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t out[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) codes4_to_f16x2<I8, 0>(in[j], out[2 * j], out[2 * j + 1]);
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// Warp-wide: write the step's rows [r0, r1) of kv head h of sequence b to present (K
// rotated when do_rotary; as E4M3 codes of an f8 cache when Q8), then make the
// generic-proxy stores visible to TMA reads.
// `staged` (shared memory, or null): the rows as [curr][D + DV] copied in at the kernel's
// start, read instead of k and v.
template <typename T, int D, int DV, bool Q8 = false, bool I8 = false>
__device__ __forceinline__ void append_rows(const DecodeArgs &a, int b, int h, int past, int r0, int r1, int lane,
                                            const uint8_t *staged = nullptr) {
  const T *kin = reinterpret_cast<const T *>(a.k), *vin = reinterpret_cast<const T *>(a.v);
  T *pk = reinterpret_cast<T *>(a.present_k), *pv = reinterpret_cast<T *>(a.present_v);
  const T *cs = reinterpret_cast<const T *>(a.cos), *sn = reinterpret_cast<const T *>(a.sin);
  constexpr int kper = D / 16;  // pairs of 8-element chunks (x[d..], x[d+D/2..]) per K row
  constexpr int vper = DV / 8;  // 8-element chunks per V row
  const int nrows = r1 - r0;
  for (int w = lane; w < nrows * (kper + vper); w += 32) {
    const bool isk = w < nrows * kper;
    const int wv = isk ? w : w - nrows * kper, per = isk ? kper : vper;
    const int rr = wv / per, c = (wv % per) * 8;
    const int pos = r0 + rr, i = pos - past;
    const size_t row = a.table ? ((size_t)a.table[(size_t)b * a.max_pages + pos / KT] * a.Hkv + h) * KT + pos % KT
                               : ((size_t)b * a.Hkv + h) * a.cap + (a.ring ? pos % a.cap : pos);
    const size_t tok = ((size_t)b * a.curr + i) * a.Hkv + h;
    const T *krow = staged ? reinterpret_cast<const T *>(staged + (size_t)i * (D + DV) * sizeof(T)) : kin + tok * D;
    const T *vrow = staged ? reinterpret_cast<const T *>(staged + (size_t)i * (D + DV) * sizeof(T)) + D
                           : vin + tok * DV;
    if (Q8) {
      uint8_t *p8 = reinterpret_cast<uint8_t *>(isk ? a.present_k : a.present_v);
      if (isk) {
        const size_t dst = row * D;
        uint4 y1 = *reinterpret_cast<const uint4 *>(krow + c);
        uint4 y2 = *reinterpret_cast<const uint4 *>(krow + D / 2 + c);
        if (a.do_rotary)
          rotate8<T>(krow + c, krow + D / 2 + c, cs + (size_t)pos * (D / 2) + c, sn + (size_t)pos * (D / 2) + c, y1,
                     y2);
        const float sc = a.k_scale[h];
        GQA_GUARD(dst + c, D / 2 + 8, a.ext.pk, a.status) {
          *reinterpret_cast<uint2 *>(p8 + dst + c) = codes8<T, I8>(y1, sc);
          *reinterpret_cast<uint2 *>(p8 + dst + D / 2 + c) = codes8<T, I8>(y2, sc);
        }
      } else {
        GQA_GUARD(row * DV + c, 8, a.ext.pv, a.status)
        *reinterpret_cast<uint2 *>(p8 + row * DV + c) =
            codes8<T, I8>(*reinterpret_cast<const uint4 *>(vrow + c), a.v_scale[h]);
      }
    } else if (isk) {
      const size_t dst = row * D;
      GQA_GUARD(dst + c, D / 2 + 8, a.ext.pk, a.status)
      if (a.do_rotary) {
        uint4 y1, y2;
        rotate8<T>(krow + c, krow + D / 2 + c, cs + (size_t)pos * (D / 2) + c, sn + (size_t)pos * (D / 2) + c, y1,
                   y2);
        *reinterpret_cast<uint4 *>(pk + dst + c) = y1;
        *reinterpret_cast<uint4 *>(pk + dst + D / 2 + c) = y2;
      } else {
        *reinterpret_cast<uint4 *>(pk + dst + c) = *reinterpret_cast<const uint4 *>(krow + c);
        *reinterpret_cast<uint4 *>(pk + dst + D / 2 + c) = *reinterpret_cast<const uint4 *>(krow + D / 2 + c);
      }
    } else {
      GQA_GUARD(row * DV + c, 8, a.ext.pv, a.status)
      *reinterpret_cast<uint4 *>(pv + row * DV + c) = *reinterpret_cast<const uint4 *>(vrow + c);
    }
  }
  fence_proxy_async_global();
  __syncwarp();
}

// Q8: the cache holds E4M3 codes (one scale per kv head for K and V) and the MMAs run on
// f16 (q converted exactly); the K scale joins the score scale and the V scale the output.
// The 16-row form converts K's codes straight into fragments and widens each warp's V rows
// to f16 in shared memory; the transposed form converts both straight from ldmatrix loads
// of the codes.
// TR: a group of at most 8 query rows runs the transposed products S^T = K Q^T and
// O^T += V^T P^T, with the warp's 16 keys (then 16 head dims of V) as the MMA's M and the
// rows as its N of 8: half the MMAs of the 16-row form, and the Q fragments stay in
// registers for the whole chunk.
template <typename T, int D, int DV, int MT, int NST, bool CL, bool MK, bool Q8 = false, bool TR = false,
          bool I8 = false>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        DecodeArgs a) {
  using L = Smem<D, DV, MT, NST, Q8>;
  using M = Mma16816<typename std::conditional<Q8, __half, T>::type>;
  static_assert(!TR || (MT == 1 && !MK && D % 32 == 0 && DV % 16 == 0), "transposed form: one 16-row tile, no mask");
  constexpr int QROWS = L::kQRows;
  constexpr int DCH = D / 8;    // 16-byte chunks per q / K row
  constexpr int VCH = DV / 8;   // 16-byte chunks per V row
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = smem + L::kStagesOff;
  uint8_t *qs = smem + L::kQOff;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
  uint64_t *xbar = full + NST;  // cluster exchange: the partials sent to this CTA have landed
  uint64_t *stallbar = xbar + 1;  // never completed (failure-path test hook)
  float *red_m = reinterpret_cast<float *>(smem + L::kRedOff);
  float *red_l = red_m + kWarps * QROWS;
  float *row_m = reinterpret_cast<float *>(smem + L::kRowOff);
  float *row_l = row_m + QROWS;
  float *sink_z = row_l + QROWS;  // sink logit of row r in the exp2 domain (0 when smooth_softmax)
  volatile int *flags = reinterpret_cast<volatile int *>(smem + L::kFlagOff);  // [0] abort, [1] last
  int *done_cnt = reinterpret_cast<int *>(smem + L::kCntOff);                 // [NST]
  int *n_issued = done_cnt + NST;

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = a.R;
  T *out = reinterpret_cast<T *>(a.out);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      done_cnt[s] = 0;
    }
    *n_issued = 0;
    mbar_init(xbar, 1);
    mbar_init(stallbar, 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  // programmatic dependent launch: the setup above may overlap the previous kernel; every
  // global read below must see its results.  The next kernel may launch right away: its
  // CTAs take SM slots this launch leaves free and wait there for this grid to complete.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  __syncthreads();
  // cluster: arrive once the barriers are initialized (released to the other CTAs); the
  // matching wait comes before the first write into another CTA's shared memory
  if constexpr (CL) cluster_arrive();

  // the step's new K/V rows of this kv head do not depend on the past length: warp 0 (the
  // one that appends them) copies them into shared memory now, so the append never waits
  // on global memory.  Every chunk of the group does this; only the last one uses them.
  uint8_t *newrows = smem + L::kNewOff;
  const bool staged = a.append && a.curr * (D + DV) * (int)sizeof(T) <= L::kNewBytes;
  if (staged && warp == 0) {
    const T *kin = reinterpret_cast<const T *>(a.k), *vin = reinterpret_cast<const T *>(a.v);
    constexpr int per_row = (D + DV) / 8;  // 16-byte chunks of one K row, then of one V row
    for (int idx = lane; idx < a.curr * per_row; idx += 32) {
      const int i = idx / per_row, ch = idx % per_row;
      const size_t tok = ((size_t)b * a.curr + i) * a.Hkv + blockIdx.y;
      cp_async16(newrows + (size_t)idx * 16, ch < D / 8 ? kin + tok * D + ch * 8 : vin + tok * DV + (ch - D / 8) * 8);
    }
    cp_async_commit();
  }
  // every exit of warp 0 first waits for those copies (none may land after the CTA is gone)
  auto drain_staged = [&] {
    if (staged && warp == 0) cp_async_wait_all();
  };

  // the past length, the sink logits and the raw query rows are loaded together: their
  // latencies overlap
  const int past = load_past(a.seqlens, a.nonpad, b, a.curr, a.cap);
  const float smul = Q8 ? a.score_mul * a.k_scale[hkv] : a.score_mul;  // the K scale joins the score scale
  const float vsc = Q8 ? a.v_scale[hkv] : 1.f;                           // and the V scale the output
  const float zsink = (threadIdx.x < R && a.head_sink) ? a.head_sink[hkv * a.G + threadIdx.x % a.G] : 0.f;
  constexpr int QITEMS = (QROWS * (DCH / 2) + kThreads - 1) / kThreads;  // chunk pairs per thread
  uint4 qraw[QITEMS][2];
#pragma unroll
  for (int u = 0; u < QITEMS; ++u) {
    const int idx = threadIdx.x + u * kThreads;
    const int r = idx / (DCH / 2), c = idx % (DCH / 2);
    qraw[u][0] = qraw[u][1] = make_uint4(0, 0, 0, 0);
    if (idx < QROWS * (DCH / 2) && r < R) {
      const T *src = reinterpret_cast<const T *>(a.q) +
                     (((size_t)b * a.curr + r / a.G) * a.Hq + hkv * a.G + r % a.G) * D;
      qraw[u][0] = *reinterpret_cast<const uint4 *>(src + c * 8);
      qraw[u][1] = *reinterpret_cast<const uint4 *>(src + D / 2 + c * 8);
    }
  }
  int st = sequence_status(past, a.curr, a.ring ? INT_MAX : a.cap, a.cap_past, a.past_separate, a.do_rotary && a.append,
                                 a.rope_len);
  if (MK && !st && (long long)past + a.curr > a.mask_keys) st = GQA_DEV_BAD_SEQLEN;  // the mask must cover every key
  if (st) {  // rejected sequence: zeros, nothing appended, reported once
    if (split == 0) {
      if (threadIdx.x == 0 && hkv == 0) report(a.status, st);
      for (int idx = threadIdx.x; idx < R * DV; idx += kThreads) {
        const int r = idx / DV, d = idx % DV, i = r / a.G, g = r % a.G;
        GQA_GUARD((((size_t)b * a.curr + i) * a.Hq + hkv * a.G + g) * DV + d, 1, a.ext.out, a.status)
        out[(((size_t)b * a.curr + i) * a.Hq + hkv * a.G + g) * DV + d] = from_f32<T>(0.f);
      }
    }
    drain_staged();
    return;
  }
  const int total = past + a.curr;
  // a ring or a paged cache starts its tiles on 64-position boundaries (a tile is then one
  // page, or never straddles the ring's wrap); the keys before the band are masked like any
  // other
  const int band_lo = a.window > 0 ? max(0, past - a.window + 1) : 0;
  const int lo = (a.ring || a.table) ? band_lo & ~(KT - 1) : band_lo;
  if (a.table) {
    // every page the group reads or writes must exist; the same decision in every CTA
    const int32_t *trow = a.table + (size_t)b * a.max_pages;
    bool bad = false;
    for (int n = lo / KT + (int)threadIdx.x; n * KT < total; n += kThreads) bad |= trow[n] < 0 || trow[n] >= a.num_pages;
    if (__syncthreads_or(bad)) {
      if (split == 0) {
        if (threadIdx.x == 0 && hkv == 0) report(a.status, GQA_DEV_BAD_PAGE);
        for (int idx = threadIdx.x; idx < R * DV; idx += kThreads) {
          const int r = idx / DV, d = idx % DV, i = r / a.G, g = r % a.G;
          GQA_GUARD((((size_t)b * a.curr + i) * a.Hq + hkv * a.G + g) * DV + d, 1, a.ext.out, a.status)
          out[(((size_t)b * a.curr + i) * a.Hq + hkv * a.G + g) * DV + d] = from_f32<T>(0.f);
        }
      }
      drain_staged();
      return;
    }
  }
  const int len = total - lo;
  const int chunk = ((len + a.splits - 1) / a.splits + KT - 1) / KT * KT;  // this group's chunk
  const int nchunks = (len + chunk - 1) / chunk;
  // a CTA past the group's last chunk has nothing to stream; in a cluster it still takes
  // part in the exchange (its rows carry m = -inf), otherwise it leaves now
  const bool idle = split >= nchunks;
  if (idle && (!CL || nchunks == 1)) {
    drain_staged();
    return;
  }
  const int c0 = lo + split * chunk;
  const int c1 = min(total, c0 + chunk);
  const int ntiles = idle ? 0 : (c1 - c0 + KT - 1) / KT;
  const int bh = b * a.Hkv + hkv;
  const bool appends = !idle && a.append && c1 > past;  // this chunk holds new rows [past, total)

  // warp 0 fills the ring; the new rows go to present before the tile that holds them.
  // (row, group) coordinates of tile t in the cache's tensor maps
  auto tile_coord = [&](int t, int &row, int &group) {
    const int k0 = c0 + t * KT;
    row = a.ring ? k0 % a.cap : k0;
    group = bh;
    if (a.table) {  // the tile is one page: rows [0, 64) of (page, kv head)
      group = a.table[(size_t)b * a.max_pages + k0 / KT] * a.Hkv + hkv;
      row = 0;
    }
  };
  auto issue = [&](int t) {
    const int s = t % NST, k0 = c0 + t * KT;
    if (appends && k0 + KT > past && k0 < total) {
      if (staged) {  // warp 0 copied them; other warps issue only after the barrier that follows
        if (warp == 0) cp_async_wait_all();
        __syncwarp();
      }
      append_rows<T, D, DV, Q8, I8>(a, b, hkv, past, max(past, k0), min(total, k0 + KT), lane,
                                staged ? newrows : nullptr);
    }
    if (lane == 0) {
      mbar_expect_tx(&full[s], L::kStageBytes);
      uint8_t *kdst = stages + s * L::kStageBytes;
      uint8_t *vdst = kdst + L::kTileBytes;
      int row, group;
      tile_coord(t, row, group);
      if constexpr (Q8) {  // [KT][128] codes each, one copy each
        tma_load_3d(kdst, &tmk, 0, row, group, &full[s]);
        tma_load_3d(vdst, &tmv, 0, row, group, &full[s]);
      } else {  // [D/64][KT][64], [DV/64][KT][64]: one copy each
        tma_load_4d(kdst, &tmk, 0, row, 0, group, &full[s]);
        tma_load_4d(vdst, &tmv, 0, row, 0, group, &full[s]);
      }
      atomicMax(n_issued, t + 1);
    }
    __syncwarp();
  };
  if (warp == 0) {
    for (int t = 0; t < min(NST, ntiles); ++t) issue(t);
  }

  // Q rows r = i*G + g (token i, q head hkv*G + g), rotated at past + i, 128B-swizzled
  {
    const T *cs = reinterpret_cast<const T *>(a.cos), *sn = reinterpret_cast<const T *>(a.sin);
    const bool rot = a.do_rotary && a.append;
#pragma unroll
    for (int u = 0; u < QITEMS; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      if (idx >= QROWS * (DCH / 2)) break;
      const int r = idx / (DCH / 2), c = idx % (DCH / 2);  // chunk c of the first half
      uint4 y1 = qraw[u][0], y2 = qraw[u][1];
      if (rot && r < R) {
        const size_t pos = (size_t)(past + r / a.G) * (D / 2);
        rotate8<T>(reinterpret_cast<const T *>(&qraw[u][0]), reinterpret_cast<const T *>(&qraw[u][1]),
                   cs + pos + c * 8, sn + pos + c * 8, y1, y2);
      }
      if (Q8) {  // the MMAs run on f16
        y1 = to_half8<T>(y1);
        y2 = to_half8<T>(y2);
      }
      const int c2 = c + DCH / 2;
      *reinterpret_cast<uint4 *>(qs + (c >> 3) * (QROWS * 128) + sw128(r, c & 7)) = y1;
      *reinterpret_cast<uint4 *>(qs + (c2 >> 3) * (QROWS * 128) + sw128(r, c2 & 7)) = y2;
    }
  }
  if (threadIdx.x < QROWS) sink_z[threadIdx.x] = zsink * kLog2e;
  drain_staged();  // the staged rows are visible to every warp after this barrier
  __syncthreads();

  float m[MT][2], l[MT][2];
  float acc[MT][DV / 8][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m[mt][h] = -INFINITY;
      l[mt][h] = 0.f;
    }
#pragma unroll
    for (int dn = 0; dn < DV / 8; ++dn)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][dn][e] = 0.f;
  }
  const uint32_t qs_u32 = smem_u32(qs);
  const int q_abs_min = past, q_abs_max = past + a.curr - 1;
  // absolute query position of this thread's rows (16*mt + lane/4 + 8h of the MMA tile), for
  // the band predicate on frontier tiles; padding rows (>= R) are marked invalid
  int qa_row[MT][2];
  bool row_ok[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = 16 * mt + (lane >> 2) + 8 * h;
      row_ok[mt][h] = row < R;
      qa_row[mt][h] = past + (row < R ? row / a.G : 0);
    }
  // transposed form: this thread's Q^T fragments (query row lane/4, head dims 16ks + 2(lane%4)
  // and + 8), its rows 2(lane%4) + j, their running maxima, sums and O^T accumulators
  uint32_t qf[TR ? D / 16 : 1][2];
  float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};
  float acct[TR ? DV / 16 : 1][4];
  int qa_t[2];
  bool ok_t[2];
  if constexpr (TR && Q8) {
    // f8 cache: k step ks covers head dims 16ks + 4t + {0, 1} (as k = 2t, 2t + 1) and
    // 16ks + 4t + {2, 3} (as k = 2t + 8, 2t + 9), the order in which K's codes arrive below
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int ch = 2 * ks + ((lane & 3) >> 1);  // 16-byte chunk of head dims 16ks + 4t .. + 3
      const uint2 w = *reinterpret_cast<const uint2 *>(qs + (ch >> 3) * (QROWS * 128) + sw128(lane >> 2, ch & 7) +
                                                       (lane & 1) * 8);
      qf[ks][0] = w.x;
      qf[ks][1] = w.y;
    }
  } else if constexpr (TR) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      const int ch = 2 * ks + (lane >> 3);  // chunks 2ks .. 2ks + 3 of query row lane % 8
      ldsm_x4(qs_u32 + (ch >> 3) * (QROWS * 128) + sw128(lane & 7, ch & 7), qf[ks][0], qf[ks][1], qf[ks + 1][0],
              qf[ks + 1][1]);
    }
  }
  if constexpr (TR) {
#pragma unroll
    for (int dm = 0; dm < DV / 16; ++dm)
#pragma unroll
      for (int e = 0; e < 4; ++e) acct[dm][e] = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int row = 2 * (lane & 3) + j;
      ok_t[j] = row < R;
      qa_t[j] = past + (row < R ? row / a.G : 0);
    }
  }
  bool aborted = false;
  int t_fail = ntiles;

  // masked kernels: this thread's mask values for a tile (rows 16*mt + lane/4 + 8h, keys
  // kb + 8n + 2*(lane%4) + {0,1}), 16 bits each, packed in pairs; loaded one tile ahead
  uint32_t mcur[MK ? MT : 1][2][2], mnext[MK ? MT : 1][2][2];
  // the mask row of each of this thread's rows (element offset of key 0), once per CTA
  long long mrow_base[MK ? MT : 1][2];
  if constexpr (MK) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = 16 * mt + (lane >> 2) + 8 * h;
        const int i = row < R ? row / a.G : 0, g = row < R ? row % a.G : 0;
        mrow_base[mt][h] = b * a.msb + (long long)(hkv * a.G + g) * a.msh + i * a.msi;
      }
  }
  auto load_mask = [&](int t, uint32_t (&mv)[MK ? MT : 1][2][2]) {
    const int kb = c0 + t * KT + 16 * warp;
    const uint32_t dflt = a.mask_kind == 1 ? 1u : 0u;  // keep / no bias where there is no row
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int key = kb + 8 * n + 2 * (lane & 3);
          uint32_t lo = dflt, hi = dflt;
          if (row_ok[mt][h]) {
            const long long base = mrow_base[MK ? mt : 0][h];
            if (a.mask_kind == 1) {
              const uint8_t *mp = reinterpret_cast<const uint8_t *>(a.mask) + base;
              if (key < a.mask_keys) lo = mp[key];
              if (key + 1 < a.mask_keys) hi = mp[key + 1];
            } else {
              const uint16_t *mp = reinterpret_cast<const uint16_t *>(a.mask) + base;
              if (key < a.mask_keys) lo = mp[key];
              if (key + 1 < a.mask_keys) hi = mp[key + 1];
            }
          }
          mv[MK ? mt : 0][n][h] = lo | (hi << 16);
        }
  };
  if constexpr (MK) {
    if (ntiles > 0) load_mask(0, mcur);
  }

  if (a.stall && ntiles > 0 &&  // failure-path test hook: a wait that nothing completes
      !__all_sync(0xffffffffu, mbar_wait(stallbar, 0, flags, a.wait_limit))) {
    aborted = true;
    t_fail = 0;
  }
  for (int t = 0; t < (aborted ? 0 : ntiles); ++t) {
    const int s = t % NST;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (t / NST) & 1, flags, a.wait_limit))) {
      aborted = true;
      t_fail = t;
      break;
    }
    const int kb = c0 + t * KT + 16 * warp;  // this warp's first key
    if constexpr (MK) {
      if (t + 1 < ntiles) load_mask(t + 1, mnext);
    }
    const uint8_t *k8 = stages + s * L::kStageBytes;  // Q8: the stage's K codes
    if constexpr (Q8 && !TR) {
      // widen the V codes of this warp's 16 keys of the stage (rows of 128 codes,
      // 128B-swizzled) to f16 in the layout of a 16-bit V tile; only this warp reads these rows
      static_assert(!Q8 || (D == 128 && DV == 128), "f8 cache: D = Dv = 128");
      const uint8_t *v8 = k8 + L::kTileBytes;
      uint8_t *vc = smem + L::kConvOff;
      const int r = 16 * warp + (lane >> 1);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int c = (lane & 1) * 4 + cc;  // codes [16c, 16c + 16) of the row
        const int e0 = 2 * c, e1 = 2 * c + 1;  // their f16 chunks
        uint4 lo, hi;
        widen16<I8>(*reinterpret_cast<const uint4 *>(v8 + r * 128 + ((c ^ (r & 7)) << 4)), lo, hi);
        *reinterpret_cast<uint4 *>(vc + (e0 >> 3) * (KT * 128) + sw128(r, e0 & 7)) = lo;
        *reinterpret_cast<uint4 *>(vc + (e1 >> 3) * (KT * 128) + sw128(r, e1 & 7)) = hi;
      }
      __syncwarp();
    }
    const uint32_t ks_u32 = smem_u32(stages + s * L::kStageBytes);
    const uint32_t vs_u32 = Q8 ? smem_u32(smem + L::kConvOff) : ks_u32 + L::kTileBytes;
    if constexpr (TR) {
      // ---- S^T = K Q^T over this warp's 16 keys: lane (g, t) = (lane/4, lane%4) holds keys
      // g and g + 8 of rows 2t and 2t + 1; even and odd k steps in two chains
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t kc[4];  // one-byte caches: the codes of two k steps
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t af[4];  // A = 16 keys x 16 head dims of K
        if constexpr (Q8) {
          // one 8x8 matrix of 16-bit pairs per 8 keys: lane (g, t) gets codes 16ks + 4t .. + 3
          // of key g (then g + 8), widened in the head-dim order of the Q fragments
          if ((ks & 1) == 0) {
            const int krow = 16 * warp + ((lane >> 3) & 1) * 8 + (lane & 7);
            const int kch = ks + (lane >> 4);
            ldsm_x4(ks_u32 + krow * 128 + ((kch ^ (krow & 7)) << 4), kc[0], kc[1], kc[2], kc[3]);
          }
          const uint32_t w0 = kc[2 * (ks & 1)], w1 = kc[2 * (ks & 1) + 1];
          codes4_to_f16x2<I8, 0>(w0, af[0], af[2]);
          codes4_to_f16x2<I8, 0>(w1, af[1], af[3]);
        } else {
          const int krow = 16 * warp + ((lane >> 4) << 3) + (lane & 7);
          const int kch = 2 * ks + ((lane >> 3) & 1);
          ldsm_x4(ks_u32 + (kch >> 3) * (KT * 128) + sw128(krow, kch & 7), af[0], af[2], af[1], af[3]);
        }
        M::run((ks & 1) ? s1 : s0, af, qf[ks][0], qf[ks][1]);
      }
      // ---- scale, softcap, band mask (frontier warps only)
      const bool edge = !(kb >= c0 && kb + 15 < c1 && (!a.causal || kb + 15 <= q_abs_min) &&
                          (a.window < 0 || q_abs_max - kb < a.window));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s0[e] + s1[e];
        x = a.cap_mul != 0.f ? tanh_fast(x * smul) * a.cap_mul : x * smul;
        if (edge) {
          const int key = kb + (lane >> 2) + 8 * (e >> 1);
          const int qa = qa_t[e & 1];
          const bool vis = ok_t[e & 1] && key >= c0 && key < c1 && (!a.causal || key <= qa) &&
                           (a.window < 0 || qa - key < a.window);
          if (!vis) x = -INFINITY;
        }
        s0[e] = x;
      }
      // ---- online softmax: a row's 16 keys sit in the 8 lanes of equal lane % 4
      float p[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float mx = fmaxf(s0[j], s0[2 + j]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (mx > mr[j] + kRescaleLog2 || (mr[j] == -INFINITY && mx != -INFINITY)) {
          const float alpha = ex2(mr[j] - mx);  // 0 while nothing was visible
          lr[j] *= alpha;
#pragma unroll
          for (int dm = 0; dm < DV / 16; ++dm) {
            acct[dm][j] *= alpha;
            acct[dm][2 + j] *= alpha;
          }
          mr[j] = mx;
        }
        const float m_use = mr[j] == -INFINITY ? 0.f : mr[j];
        p[j] = ex2(s0[j] - m_use);
        p[2 + j] = ex2(s0[2 + j] - m_use);
        lr[j] += p[j] + p[2 + j];
      }
      // P^T as the B operand (keys 2t, 2t + 1 (+ 8) of row g): each 8x8 block transposed
      const uint32_t pb0 = movm_t(M::pack(p[0], p[1])), pb1 = movm_t(M::pack(p[2], p[3]));
      if (kb + 16 > total) {
        const int first = max(0, total - kb);
        if constexpr (Q8) {  // the V codes in the stage (code 0 is +0)
          for (int idx = lane; idx < (16 - first) * 8; idx += 32) {
            const int r = 16 * warp + first + idx / 8, ch = idx % 8;
            *reinterpret_cast<uint4 *>(stages + s * L::kStageBytes + L::kTileBytes + r * 128 + ((ch ^ (r & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
        } else {
          for (int idx = lane; idx < (16 - first) * VCH; idx += 32) {
            const int r = 16 * warp + first + idx / VCH, ch = idx % VCH;
            *reinterpret_cast<uint4 *>(stages + s * L::kStageBytes + L::kTileBytes + (ch >> 3) * (KT * 128) +
                                       sw128(r, ch & 7)) = make_uint4(0, 0, 0, 0);
          }
        }
        __syncwarp();
      }
      // ---- O^T += V^T P^T: A = 16 head dims x 16 keys of V (transposing loads)
      if constexpr (Q8) {
        // one transposed 8x8 matrix of 16-bit code pairs per 8 keys and 16 head dims: lane
        // (g, t) gets codes 16dm + 2g, 2g + 1 of keys 2t and 2t + 1; a byte permute pairs
        // them by head dim, so A's row g is head dim 16dm + 2g and row g + 8 is 16dm + 2g + 1
        const uint32_t vc_u32 = ks_u32 + L::kTileBytes;
#pragma unroll
        for (int dm = 0; dm < DV / 16; dm += 2) {
          uint32_t w[4];
          const int vrow = 16 * warp + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int vch = dm + (lane >> 4);
          ldsm_x4_t(vc_u32 + vrow * 128 + ((vch ^ (vrow & 7)) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t af[4];
            codes4_to_f16x2<I8, 1>(w[2 * h], af[0], af[1]);
            codes4_to_f16x2<I8, 1>(w[2 * h + 1], af[2], af[3]);
            M::run(acct[dm + h], af, pb0, pb1);
          }
        }
      } else {
#pragma unroll
        for (int dm = 0; dm < DV / 16; ++dm) {
          uint32_t af[4];
          const int vrow = 16 * warp + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int vch = 2 * dm + (lane >> 4);
          ldsm_x4_t(vs_u32 + (vch >> 3) * (KT * 128) + sw128(vrow, vch & 7), af[0], af[2], af[1], af[3]);
          M::run(acct[dm], af, pb0, pb1);
        }
      }
    } else {
      // ---- S = Q K^T over this warp's 16 keys, the k steps split over two independent
      // accumulator chains (even and odd steps) that are added at the end
      float sacc[MT][2][4], sodd[MT][2][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mt][n][e] = sodd[mt][n][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t kb0, kb1, kb2, kb3;
        if constexpr (Q8) {
          // the B fragments straight from the codes: key row 16*warp + lane/4 (+8), head dims
          // 16*ks + 2*(lane%4) (+8), i.e. a pair of neighbouring bytes of 16-byte chunk ks of
          // the row, one pair conversion each
          const int r0 = 16 * warp + (lane >> 2), o = 2 * (lane & 3);
          const uint8_t *c0 = k8 + r0 * 128 + ((ks ^ (r0 & 7)) << 4) + o;
          const uint8_t *c1 = c0 + 8 * 128;  // row r0 + 8: the same swizzle phase
          kb0 = codes2_to_f16x2<I8>(*reinterpret_cast<const uint16_t *>(c0));
          kb1 = codes2_to_f16x2<I8>(*reinterpret_cast<const uint16_t *>(c0 + 8));
          kb2 = codes2_to_f16x2<I8>(*reinterpret_cast<const uint16_t *>(c1));
          kb3 = codes2_to_f16x2<I8>(*reinterpret_cast<const uint16_t *>(c1 + 8));
        } else {
          const int krow = 16 * warp + ((lane >> 4) << 3) + (lane & 7);
          const int kch = 2 * ks + ((lane >> 3) & 1);
          ldsm_x4(ks_u32 + (kch >> 3) * (KT * 128) + sw128(krow, kch & 7), kb0, kb1, kb2, kb3);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t af[4];
          const int qrow = 16 * mt + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int qch = 2 * ks + (lane >> 4);
          ldsm_x4(qs_u32 + (qch >> 3) * (QROWS * 128) + sw128(qrow, qch & 7), af[0], af[1], af[2], af[3]);
          M::run((ks & 1) ? sodd[mt][0] : sacc[mt][0], af, kb0, kb1);
          M::run((ks & 1) ? sodd[mt][1] : sacc[mt][1], af, kb2, kb3);
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mt][n][e] += sodd[mt][n][e];

      // ---- scale, softcap, band mask (only on warps whose keys cross a frontier)
      const bool edge = !(kb >= c0 && kb + 15 < c1 && (!a.causal || kb + 15 <= q_abs_min) &&
                          (a.window < 0 || q_abs_max - kb < a.window));
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = sacc[mt][n][e];
            bool dropped = false;
            if constexpr (MK) {
              const uint32_t bits = (mcur[mt][n][e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
              if (a.mask_kind == 1) {
                dropped = bits == 0;
              } else {
                T bv;
                *reinterpret_cast<uint16_t *>(&bv) = (uint16_t)bits;
                x = fmaf(to_f32(bv), a.mask_mul, x);  // the bias joins before the scale and softcap
              }
            }
            x = a.cap_mul != 0.f ? tanh_fast(x * smul) * a.cap_mul : x * smul;
            if (dropped) x = -INFINITY;
            if (edge) {
              const int key = kb + 8 * n + 2 * (lane & 3) + (e & 1);
              const int qa = qa_row[mt][e >> 1];
              const bool vis = row_ok[mt][e >> 1] && key >= c0 && key < c1 && (!a.causal || key <= qa) &&
                               (a.window < 0 || qa - key < a.window);
              if (!vis) x = -INFINITY;
            }
            sacc[mt][n][e] = x;
          }

      // ---- online softmax, reference max moved lazily (rows lane/4 and lane/4 + 8)
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
          if (mx > m[mt][h] + kRescaleLog2 || (m[mt][h] == -INFINITY && mx != -INFINITY)) {
            const float alpha = ex2(m[mt][h] - mx);  // 0 while nothing was visible
            l[mt][h] *= alpha;
#pragma unroll
            for (int dn = 0; dn < DV / 8; ++dn) {
              acc[mt][dn][2 * h] *= alpha;
              acc[mt][dn][2 * h + 1] *= alpha;
            }
            m[mt][h] = mx;
          }
          const float m_use = m[mt][h] == -INFINITY ? 0.f : m[mt][h];
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float pv = ex2(sacc[mt][n][2 * h + e] - m_use);
              p[n][2 * h + e] = pv;
              l[mt][h] += pv;
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
        for (int idx = lane; idx < (16 - first) * VCH; idx += 32) {
          const int r = 16 * warp + first + idx / VCH, ch = idx % VCH;
          *reinterpret_cast<uint4 *>((Q8 ? smem + L::kConvOff : stages + s * L::kStageBytes + L::kTileBytes) +
                                     (ch >> 3) * (KT * 128) +
                                     sw128(r, ch & 7)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }

      // ---- O += P V over this warp's 16 keys
#pragma unroll
      for (int dd = 0; dd < DV / 16; ++dd) {
        uint32_t v0, v1, v2, v3;
        const int vrow = 16 * warp + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int vch = 2 * dd + (lane >> 4);
        ldsm_x4_t(vs_u32 + (vch >> 3) * (KT * 128) + sw128(vrow, vch & 7), v0, v1, v2, v3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          M::run(acc[mt][2 * dd], pa[mt], v0, v1);
          M::run(acc[mt][2 * dd + 1], pa[mt], v2, v3);
        }
      }
    }
    if (kb + 16 > total) fence_proxy_async_smem();
    __syncwarp();
    // the last of the four warps to finish with the stage refills it: nobody waits for the
    // others (the count only grows; every fourth arrival is a tile's last)
    if (t + NST < ntiles) {
      int last = 0;
      if (lane == 0) {
        __threadfence_block();  // this warp's reads of the stage are ordered before its count
        last = (atomicAdd(&done_cnt[s], 1) % kWarps) == kWarps - 1;
        if (last) __threadfence_block();
      }
      if (__shfl_sync(0xffffffffu, last, 0)) issue(t + NST);
    }
    if constexpr (MK) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          mcur[mt][n][0] = mnext[mt][n][0];
          mcur[mt][n][1] = mnext[mt][n][1];
        }
    }
  }

  drain_staged();  // long complete by now

  // -------------------------------------------------------------- merge the 4 warps
  // per-warp row statistics (outside the stages: safe while aborted copies still land)
  if constexpr (TR) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float lv = lr[j];
      lv += __shfl_xor_sync(0xffffffffu, lv, 4);
      lv += __shfl_xor_sync(0xffffffffu, lv, 8);
      lv += __shfl_xor_sync(0xffffffffu, lv, 16);
      if (lane < 4) {
        const int row = 2 * lane + j;
        red_m[warp * QROWS + row] = mr[j];
        red_l[warp * QROWS + row] = lv;
        red_m[warp * QROWS + 8 + row] = -INFINITY;  // rows 8-15 of the tile: none
        red_l[warp * QROWS + 8 + row] = 0.f;
      }
    }
  } else {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float lv = l[mt][h];
        lv += __shfl_xor_sync(0xffffffffu, lv, 1);
        lv += __shfl_xor_sync(0xffffffffu, lv, 2);
        if ((lane & 3) == 0) {
          const int row = 16 * mt + (lane >> 2) + 8 * h;
          red_m[warp * QROWS + row] = m[mt][h];
          red_l[warp * QROWS + row] = lv;
        }
      }
  }
  // one decision for the whole CTA (a timed-out wait anywhere aborts it), taken by the
  // barrier that publishes the statistics
  aborted = __syncthreads_or(aborted || flags[0] != 0);
  if (aborted) {
    // copies in flight must land before the CTA exits; take part in the ticket (or the
    // cluster exchange, with no visible key) so the group stays consistent, write nothing
    if (threadIdx.x == 0) {
      volatile int no_abort = 0;
      for (int t = t_fail; t < min(*n_issued, t_fail + NST); ++t) mbar_wait(&full[t % NST], (t / NST) & 1, &no_abort);
      report(a.status, GQA_DEV_TIMEOUT);
      if (!CL && nchunks > 1) {
        __threadfence();
        GQA_GUARD(bh, 1, a.ext.tickets, a.status) {
          const int old = atomicAdd(&a.tickets[bh], 1);
          if (old == nchunks - 1) a.tickets[bh] = 0;
        }
      }
    }
    if constexpr (CL) {
      if (nchunks == 1) return;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) m[mt][0] = m[mt][1] = -INFINITY;
      mr[0] = mr[1] = -INFINITY;
      for (int i = threadIdx.x; i < kWarps * QROWS; i += kThreads) red_m[i] = -INFINITY;
      __syncthreads();  // uniform branch; thread 0 has drained the copies
    } else {
      return;
    }
  }
  // cluster exchange: into the dedicated region when the partials fit (no barrier needed
  // now: every CTA arrived at the start), else into the stages, which peers may only write
  // once every CTA of the cluster has finished streaming (a second barrier phase)
  const int S_cl = gridDim.x, n4_cl = R * (DV / 4), per_cl = (n4_cl + S_cl - 1) / S_cl;
  const bool rcv_own = CL && S_cl * per_cl * 16 + S_cl * QROWS * 8 <= L::kRcvBytes;
  if (CL && nchunks > 1 && !rcv_own) {
    cluster_wait();            // first phase: completed at the start
    cluster_arrive_relaxed();  // this CTA's stages are free (nothing in flight)
  }
  // row statistics over the four warps (threads < QROWS), and every warp's accumulator
  // rescaled to the row maximum (each lane takes the maximum of its own rows from the warps'
  // maxima) in its own region of the now free stages; all threads then sum the four regions
  // in a fixed order (deterministic)
  if (threadIdx.x < QROWS) {
    const int row = threadIdx.x;
    float mm = -INFINITY;
    for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, red_m[w * QROWS + row]);
    const float mu = mm == -INFINITY ? 0.f : mm;
    float ll = 0.f;
    for (int w = 0; w < kWarps; ++w) ll += red_l[w * QROWS + row] * ex2(red_m[w * QROWS + row] - mu);
    row_m[row] = mm;
    row_l[row] = ll;
  }
  constexpr int AST = L::kAccStride;
  float *wacc = reinterpret_cast<float *>(stages);  // [kWarps][QROWS][AST]
  if constexpr (TR) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int row = 2 * (lane & 3) + j;
      if (row >= R) continue;  // padding rows are never read
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, red_m[w * QROWS + row]);
      const float f = ex2(mr[j] - (mm == -INFINITY ? 0.f : mm));
      if constexpr (Q8) {  // head dims 16dm + 2(lane/4) and + 1
        float *dst = wacc + ((size_t)warp * QROWS + row) * AST + 2 * (lane >> 2);
#pragma unroll
        for (int dm = 0; dm < DV / 16; ++dm)
          *reinterpret_cast<float2 *>(dst + 16 * dm) = make_float2(acct[dm][j] * f, acct[dm][2 + j] * f);
      } else {  // head dims 16dm + lane/4 and + 8
        float *dst = wacc + ((size_t)warp * QROWS + row) * AST + (lane >> 2);
#pragma unroll
        for (int dm = 0; dm < DV / 16; ++dm) {
          dst[16 * dm] = acct[dm][j] * f;
          dst[16 * dm + 8] = acct[dm][2 + j] * f;
        }
      }
    }
  } else {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = 16 * mt + (lane >> 2) + 8 * h;
        if (row >= R) continue;  // padding rows of the MMA tile are never read
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, red_m[w * QROWS + row]);
        const float f = ex2(m[mt][h] - (mm == -INFINITY ? 0.f : mm));
        float *dst = wacc + ((size_t)warp * QROWS + row) * AST + 2 * (lane & 3);
#pragma unroll
        for (int dn = 0; dn < DV / 8; ++dn)
          *reinterpret_cast<float2 *>(dst + 8 * dn) = make_float2(acc[mt][dn][2 * h] * f, acc[mt][dn][2 * h + 1] * f);
      }
  }
  __syncthreads();
  auto merged = [&](int idx4) {  // float4 idx4 of the CTA's [R][DV] accumulator
    const float4 *w4 = reinterpret_cast<const float4 *>(wacc) + (idx4 / (DV / 4)) * (AST / 4) + idx4 % (DV / 4);
    float4 v = w4[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      const float4 u = w4[w * (QROWS * AST / 4)];
      v.x += u.x;
      v.y += u.y;
      v.z += u.z;
      v.w += u.w;
    }
    return v;
  };

  if (nchunks == 1) {
    // ------------------------------------------------------------ finish in place
    for (int idx = threadIdx.x; idx < R * (DV / 4); idx += kThreads) {
      const int r = idx / (DV / 4), d4 = idx % (DV / 4);
      const int i = r / a.G, g = r % a.G, hq = hkv * a.G + g;
      const float mm = row_m[r];
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 1.f;
      if (mm != -INFINITY) {
        float top = mm, sink_term = 0.f;
        if (a.has_sink) {
          const float z = sink_z[r];
          top = fmaxf(mm, z);
          sink_term = ex2(z - top);
        }
        const float f = ex2(mm - top);
        num = merged(idx);
        num.x *= f;
        num.y *= f;
        num.z *= f;
        num.w *= f;
        den = row_l[r] * f + sink_term;
      }
      T *o = out + (((size_t)b * a.curr + i) * a.Hq + hq) * DV + d4 * 4;
      const float inv = __frcp_rn(den) * vsc;
      GQA_GUARD((((size_t)b * a.curr + i) * a.Hq + hq) * DV + d4 * 4, 4, a.ext.out, a.status)
      store4(o, num.x * inv, num.y * inv, num.z * inv, num.w * inv);
    }
    return;
  }

  if (CL) {
    // ------------------------------------------------------------ cluster exchange
    // the group's chunks are the CTAs of one cluster.  CTA `rank` owns float4 slice
    // [rank * per, (rank + 1) * per) of the group's [R][DV] output; every CTA pushes its
    // (m, l) rows and the matching slice of its accumulator into the owner's shared memory
    // (after the wacc regions) with asynchronous stores that count down the owner's xbar.
    // The owner waits for exactly those bytes and combines its slice from local data; once
    // they have landed nothing else writes to or reads from its shared memory, so it may exit
    const int S = S_cl, rank = split;
    const int n4 = n4_cl, per = per_cl;
    // [S][per] float4 slices, then [S][QROWS] (m, l)
    float *rcv = rcv_own ? reinterpret_cast<float *>(smem + L::kRcvOff) : wacc + kWarps * QROWS * AST;
    float2 *rcv_ml = reinterpret_cast<float2 *>(rcv + (rcv_own ? S * per * 4 : QROWS * DV + 4 * kMaxCluster));
    // dedicated region: the start's phase (every peer's barriers are initialized); stages:
    // the second phase (every peer has finished streaming)
    cluster_wait();
    const uint32_t rcv_s = smem_u32(rcv), rml_s = smem_u32(rcv_ml), xb_s = smem_u32(xbar);
    for (int t = threadIdx.x; t < S * R; t += kThreads) {
      const int k = t / R, r = t % R;
      cluster_st_async2(cluster_map(rml_s + 8 * (rank * QROWS + r), k), row_m[r], row_l[r], cluster_map(xb_s, k));
    }
    for (int idx = threadIdx.x; idx < n4; idx += kThreads) {
      const int dst = idx / per;
      cluster_st_async4(cluster_map(rcv_s + 16 * (rank * per + idx - dst * per), dst), merged(idx),
                        cluster_map(xb_s, dst));
    }
    const int lo4 = rank * per, hi4 = min(n4, lo4 + per);
    if (threadIdx.x == 0) mbar_expect_tx(xbar, S * (max(0, hi4 - lo4) * 16 + R * 8));
    if (!mbar_wait_cluster(xbar, 0)) {  // a peer never delivered: nothing valid to combine
      if (threadIdx.x == 0) report(a.status, GQA_DEV_TIMEOUT);
      return;
    }
    // each output float4 weighs the chunks of its row itself: no second pass, no barrier
    const float4 *rcv4 = reinterpret_cast<const float4 *>(rcv);
    for (int idx = lo4 + threadIdx.x; idx < hi4; idx += kThreads) {
      const int r = idx / (DV / 4), d4 = idx % (DV / 4);
      const int i = r / a.G, g = r % a.G, hq = hkv * a.G + g;
      float mk[kMaxCluster];
      float top = -INFINITY;
#pragma unroll
      for (int k = 0; k < kMaxCluster; ++k) {
        mk[k] = k < S ? rcv_ml[k * QROWS + r].x : -INFINITY;
        top = fmaxf(top, mk[k]);
      }
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 1.f;  // no visible key: the sums stay 0
      if (top != -INFINITY) {
        float ll = 0.f;
        if (a.has_sink) {
          const float z = sink_z[r];
          top = fmaxf(top, z);
          ll = ex2(z - top);
        }
#pragma unroll
        for (int k = 0; k < kMaxCluster; ++k) {
          if (mk[k] == -INFINITY) continue;  // past the cluster, or a chunk without a visible key
          const float f = ex2(mk[k] - top);
          ll += rcv_ml[k * QROWS + r].y * f;
          const float4 v = rcv4[k * per + idx - lo4];
          sum.x += v.x * f;
          sum.y += v.y * f;
          sum.z += v.z * f;
          sum.w += v.w * f;
        }
        den = ll;
      }
      T *o = out + (((size_t)b * a.curr + i) * a.Hq + hq) * DV + d4 * 4;
      const float inv = __frcp_rn(den) * vsc;
      GQA_GUARD((((size_t)b * a.curr + i) * a.Hq + hq) * DV + d4 * 4, 4, a.ext.out, a.status)
      store4(o, sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
    }
    return;  // nothing reads this CTA's shared memory any more
  }

  // -------------------------------------------------------------- write the partial
  const size_t gbase = (size_t)bh * a.splits * R;
  {
    const size_t base = gbase + (size_t)split * R;
    float4 *pacc = reinterpret_cast<float4 *>(a.part_acc + base * DV);
    for (int idx = threadIdx.x; idx < R * DV / 4; idx += kThreads) {
      GQA_GUARD(base * DV + 4 * (size_t)idx, 4, a.ext.part_acc, a.status)
      pacc[idx] = merged(idx);
    }
    for (int r = threadIdx.x; r < R; r += kThreads)
      GQA_GUARD(2 * (base + r), 2, a.ext.part_ml, a.status)
      reinterpret_cast<float2 *>(a.part_ml)[base + r] = make_float2(row_m[r], row_l[r]);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int old = 0;
    GQA_GUARD(bh, 1, a.ext.tickets, a.status)
    old = atomicAdd(&a.tickets[bh], 1);
    flags[1] = old == nchunks - 1;
  }
  __syncthreads();
  if (!flags[1]) return;

  // -------------------------------------------------------------- last CTA: combine
  __threadfence();
  if (threadIdx.x == 0) {
    GQA_GUARD(bh, 1, a.ext.tickets, a.status)
    a.tickets[bh] = 0;
  }
  // chunk statistics staged in shared memory with all loads in flight at once
  float *cm = reinterpret_cast<float *>(stages);  // [nchunks][R] max, then scale factor
  float *cl = cm + a.splits * R;                    // [nchunks][R] sum
  for (int idx = threadIdx.x; idx < nchunks * R; idx += kThreads) {
    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.part_ml) + gbase + idx);
    cm[idx] = ml.x;
    cl[idx] = ml.y;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += kThreads) {
    float mm = -INFINITY;
    for (int c = 0; c < nchunks; ++c) mm = fmaxf(mm, cm[c * R + r]);
    float top = mm, sink_term = 0.f;
    if (mm != -INFINITY && a.has_sink) {
      const float z = sink_z[r];
      top = fmaxf(mm, z);
      sink_term = ex2(z - top);
    }
    float ll = sink_term;
    for (int c = 0; c < nchunks; ++c) {
      const float f = mm == -INFINITY ? 0.f : ex2(cm[c * R + r] - top);  // 0 for empty chunks
      ll += cl[c * R + r] * f;
      cm[c * R + r] = f;
    }
    row_l[r] = mm == -INFINITY ? 0.f : ll;
  }
  __syncthreads();
  // chunk-outer: every thread keeps its outputs in registers and issues one independent
  // load per output per chunk
  constexpr int kPer = (MT * 16 * DV / 4 + kThreads - 1) / kThreads;
  float4 sum[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) sum[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 *pa4 = reinterpret_cast<const float4 *>(a.part_acc + gbase * DV);
#pragma unroll 4
  for (int c = 0; c < nchunks; ++c) {
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      if (idx < R * (DV / 4)) {
        const float f = cm[c * R + idx / (DV / 4)];
        const float4 v = __ldcg(pa4 + (size_t)c * R * (DV / 4) + idx);
        sum[u].x += v.x * f;
        sum[u].y += v.y * f;
        sum[u].z += v.z * f;
        sum[u].w += v.w * f;
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int idx = threadIdx.x + u * kThreads;
    if (idx >= R * (DV / 4)) continue;
    const int r = idx / (DV / 4), d4 = idx % (DV / 4);
    const int i = r / a.G, g = r % a.G, hq = hkv * a.G + g;
    const float den = row_l[r] > 0.f ? row_l[r] : 1.f;  // no visible key: the sums are 0
    T *o = out + (((size_t)b * a.curr + i) * a.Hq + hq) * DV + d4 * 4;
    const float inv = __frcp_rn(den) * vsc;
    GQA_GUARD((((size_t)b * a.curr + i) * a.Hq + hq) * DV + d4 * 4, 4, a.ext.out, a.status)
    store4(o, sum[u].x * inv, sum[u].y * inv, sum[u].z * inv, sum[u].w * inv);
  }
}

template <typename T, int D, int DV, int MT, int NST, bool CL, bool MK, bool Q8 = false, bool TR = false,
          bool I8 = false>
gqa_status launch_cfg(const Call &c, const DecodePlan &dp, const DecodeArgs &a) {
  using L = Smem<D, DV, MT, NST, Q8>;
  static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
  CUtensorMap tk, tv;
  // contiguous or ring: [B*Hkv][cap][D] and [..][DV]; paged: [num_pages*Hkv][64][D]
  const bool paged = c.block_table != nullptr;
  const long long outer = paged ? (long long)c.num_pages * c.p.kv_heads : (long long)c.p.batch * c.p.kv_heads;
  const int rows = paged ? KT : c.p.cap_present;
  if (Q8) {  // [B*Hkv][cap][128] codes: a 64-row box of whole 128-byte rows
    if (!encode_kv8_map(&tk, c.present_k, D, rows, outer, KT)) return GQA_ERR_CUDA;
    if (!encode_kv8_map(&tv, c.present_v, DV, rows, outer, KT)) return GQA_ERR_CUDA;
  } else {
    if (!encode_kv_tile_map(&tk, c.present_k, D, rows, outer, KT, 2)) return GQA_ERR_CUDA;
    if (!encode_kv_tile_map(&tv, c.present_v, DV, rows, outer, KT, 2)) return GQA_ERR_CUDA;
  }
  auto kern = decode_split_kernel<T, D, DV, MT, NST, CL, MK, Q8, TR, I8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess)
    return GQA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dp.splits, c.p.kv_heads, c.p.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (CL) {  // the chunks of one group form one cluster
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = dp.splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  if (cudaLaunchKernelEx(&cfg, kern, tk, tv, a) != cudaSuccess) return GQA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

template <typename T, bool CL, bool MK, bool MIXED, bool Q8, bool I8>
gqa_status dispatch(const Call &c, const DecodePlan &dp, const DecodeArgs &a);

template <typename T, bool MK, bool MIXED, bool Q8 = false, bool I8 = false>
gqa_status launch_t(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  const gqa_params &p = c.p;
  DecodeArgs a;
  a.q = c.q_in;
  a.k = c.k;
  a.v = c.v;
  a.cos = c.cos;
  a.sin = c.sin;
  a.present_k = c.present_k;
  a.present_v = c.present_v;
  a.out = c.out;
  a.seqlens = c.seqlens;
  a.nonpad = c.nonpad;
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
  a.ring = p.kv_ring;
  a.table = c.block_table;
  a.max_pages = c.max_pages;
  a.num_pages = c.num_pages;
  a.mask = c.mask;
  a.mask_kind = c.mask_kind;
  a.mask_keys = c.mask_keys;
  a.msb = c.mask_sb;
  a.msh = c.mask_sh;
  a.msi = c.mask_si;
  a.mask_mul = 1.f / p.scale;
  a.cap_past = p.cap_past;
  a.past_separate = c.past_separate;
  a.rope_len = p.rope_len;
  a.do_rotary = p.do_rotary;
  a.append = c.append;
  a.window = p.window;
  a.causal = p.causal;
  a.splits = dp.splits;
  a.has_sink = (c.head_sink != nullptr) || p.smooth_softmax;
  if (p.softcap > 0.f) {
    a.score_mul = p.scale / p.softcap;
    a.cap_mul = p.softcap * kLog2e;
  } else {
    a.score_mul = p.scale * kLog2e;
    a.cap_mul = 0.f;
  }
  a.k_scale = c.k_scale;
  a.v_scale = c.v_scale;
  a.wait_limit = c.wait_limit > 0 ? c.wait_limit : kWaitLimitCycles;
  a.stall = c.stall;
#ifdef GQA_BOUNDS_CHECK
  a.ext = extents_of(c, wl);
#endif
  if (dp.cluster) return dispatch<T, true, MK, MIXED, Q8, I8>(c, dp, a);
  return dispatch<T, false, MK, MIXED, Q8, I8>(c, dp, a);
}

// (D, DV, MT, NST): equal head dims (MIXED false; at D = 128 three 32 KB stages, two CTAs per
// SM) or V head dim != Q/K head dim (MIXED true, up to 32 query rows per group; four stages
// of 24 KB)
template <typename T, bool CL, bool MK, bool MIXED, bool Q8, bool I8>
gqa_status dispatch(const Call &c, const DecodePlan &dp, const DecodeArgs &a) {
  const int D = c.p.head_dim, DV = c.Dv;
  if constexpr (Q8) {  // f8 cache: D = Dv = 128, five 16 KB stages and a 16 KB f16 V tile
    if (D == 128 && DV == 128 && !MK && !MIXED) {
      if (dp.mtiles == 1 && dp.rows <= 8) return launch_cfg<T, 128, 128, 1, 5, CL, false, true, true, I8>(c, dp, a);
      if (dp.mtiles == 1) return launch_cfg<T, 128, 128, 1, 5, CL, false, true, false, I8>(c, dp, a);
      if (dp.mtiles == 2) return launch_cfg<T, 128, 128, 2, 5, CL, false, true, false, I8>(c, dp, a);
    }
  } else if constexpr (!MIXED) {
    if (D == 128 && DV == 128) {
      if constexpr (!MK) {  // at most 8 rows: the transposed form
        if (dp.rows <= 8) return launch_cfg<T, 128, 128, 1, 3, CL, false, false, true>(c, dp, a);
      }
      if (dp.mtiles == 1) return launch_cfg<T, 128, 128, 1, 3, CL, MK>(c, dp, a);
      if (dp.mtiles == 2) return launch_cfg<T, 128, 128, 2, 3, CL, MK>(c, dp, a);
    } else if (D == 64 && DV == 64) {
      if constexpr (!MK) {  // at most 8 rows: the transposed form
        if (dp.rows <= 8) return launch_cfg<T, 64, 64, 1, 6, CL, false, false, true>(c, dp, a);
      }
      if (dp.mtiles == 1) return launch_cfg<T, 64, 64, 1, 6, CL, MK>(c, dp, a);
      if (dp.mtiles == 2) return launch_cfg<T, 64, 64, 2, 6, CL, MK>(c, dp, a);
      if (dp.mtiles == 3) return launch_cfg<T, 64, 64, 3, 6, CL, MK>(c, dp, a);
      if (dp.mtiles == 4) return launch_cfg<T, 64, 64, 4, 6, CL, MK>(c, dp, a);
    }
  } else {
    if (D == 128 && DV == 64) {
      if constexpr (!MK) {  // at most 8 rows: the transposed form
        if (dp.rows <= 8) return launch_cfg<T, 128, 64, 1, 4, CL, false, false, true>(c, dp, a);
      }
      if (dp.mtiles == 1) return launch_cfg<T, 128, 64, 1, 4, CL, MK>(c, dp, a);
      if (dp.mtiles == 2) return launch_cfg<T, 128, 64, 2, 4, CL, MK>(c, dp, a);
    } else if (D == 64 && DV == 128) {
      if constexpr (!MK) {  // at most 8 rows: the transposed form
        if (dp.rows <= 8) return launch_cfg<T, 64, 128, 1, 4, CL, false, false, true>(c, dp, a);
      }
      if (dp.mtiles == 1) return launch_cfg<T, 64, 128, 1, 4, CL, MK>(c, dp, a);
      if (dp.mtiles == 2) return launch_cfg<T, 64, 128, 2, 4, CL, MK>(c, dp, a);
    }
  }
  return GQA_ERR_UNSUPPORTED;
}

// The decode launch for one dtype switch; each .cu file instantiates one (MK, MIXED) pair
// (masked or not, equal or different head dims), so the sets compile in parallel.
template <bool MK, bool MIXED, bool Q8 = false, bool I8 = false>
gqa_status launch_decode_split_impl(const Call &c, const DecodePlan &dp, const WsLayout &wl) {
  switch (c.p.dtype) {
    case GQA_F16: return launch_t<__half, MK, MIXED, Q8, I8>(c, dp, wl);
    case GQA_BF16: return launch_t<__nv_bfloat16, MK, MIXED, Q8, I8>(c, dp, wl);
  }
  return GQA_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace gqa

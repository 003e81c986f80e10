// prefill_tc.cuh -- K2: flash-attention forward on the 5th-generation tensor cores.
//
// onnx-light-cpu "Attention Kernel Design": streaming online softmax over KV blocks with
// a running max, denominator and unnormalized output per row; causal/padding frontiers
// skip whole blocks ("Compute paths"); fp32 accumulation, output narrowed once; a fully
// masked row gives zeros ("Scheduling, precision, and invariants").  OpenVINO PR #37423:
// window band in absolute positions ("Sliding window"); the sink joins the denominator
// ("smooth_softmax / head_sink").  tract PR #2645 ("What changed"): bottom-right band.
//
// One CTA = one tile of 128 query rows of TWO q heads of the same kv group (they share
// every K/V tile and have the same band), 12 warps, one CTA per SM (about 198 KB of shared
// memory and all 512 TMEM columns: S_A, S_B, O_A, O_B, 128 columns each).  Roles:
//   warp 0  producer: TMA loads of both Q tiles once, then K tiles (128 keys, 128B swizzle)
//           through a ring of kKStages and V tiles through two stages, each released by a
//           tcgen05.commit of the MMAs that read it
//   warp 1  TMEM owner + MMA issuer (one thread): S = Q K^T (M=128, N=128, K=D) into TMEM
//           per head, then O += P V (N = DV, the V head dim) with P read from TMEM (it
//           overwrites the first columns of S in place as packed pairs); the issue order
//           S_A(t), S_B(t), PV_A(t-1), ... interleaves the heads so one head's softmax
//           overlaps the other head's MMAs
//   warp 2  mask producer (masked kernels only; idle otherwise), warp 3 idle
//   warps 4-7 and 8-11  one softmax warpgroup per head: thread = one TMEM lane = one query
//           row; tcgen05.ld of S, band mask on frontier tiles only, scale/softcap, exp2
//           online softmax with a lazily rescaled reference max, P back to TMEM with
//           tcgen05.st, final O / l epilogue
// KV tiles outside [window low, causal high] are never visited; only tiles that cross a
// frontier evaluate the per-element predicate.
// The sink starts the running state: m = z*log2(e), l = 1, so it is counted exactly once.
//
// With an attention mask (MK = 1 boolean keep flags, 2 additive values per head, 3 additive
// values shared by the heads; onnx-light-cpu "Layouts and semantics"), warp 2 streams the
// mask's [128 rows x 128 keys] tile into shared memory by TMA, one buffer per head (MK 1,
// 2) or one for both (MK 3) released by the softmax that reads it; the softmax applies it
// to S before the row maximum.  Key tiles then start on 16-key boundaries (the TMA rule for
// the mask's inner coordinate); the extra keys lie outside the band.  With per-head
// additive tiles and D = 128 the K ring has one stage, to make room.
#pragma once
#include <float.h>
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace gqa {
namespace {

constexpr int BM = 128;       // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;       // keys per tile
constexpr int kThreads = 384; // 12 warps: producer, MMA, 2 spare, 2 softmax warpgroups
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by more than 2^8

struct PrefillArgs {
  void *out;
  const int32_t *seqlens;
  const int64_t *nonpad;  // padded cache: valid keys per sequence (replaces seqlens)
  const float *head_sink;
  int32_t *status;
  int Hq, Hkv, G, curr, cap, cap_past, past_separate, rope_len, do_rotary, window, causal, has_sink;
  float score_mul, cap_mul;  // as in the decode kernel
  // attention mask (MK > 0): keys < mask_keys; a broadcast dimension reads coordinate 0
  int mask_keys, mask_bcast_b, mask_bcast_h, mask_bcast_i;
  float bias_mul;  // 1 / scale: an additive value joins the raw dot product before scaling
  long long wait_limit;  // SM cycles after which a pipeline wait gives up
  int stall;             // test hook: the first wait is on a barrier nothing completes
  // ring cache: position p in row p % cap (cap a multiple of 128); paged cache: pools
  // [num_pages * Hkv][64][D], table [B][max_pages] names the page of positions [64n, 64n + 64)
  int ring;
  const int32_t *table;
  int max_pages, num_pages;
  // boolean mask (MK 1): the block map of the mask, or null.  Bit c of word w of row
  // ((bm * bm_heads + hm) * bm_qtiles + qm) says whether any key of 16-key chunk 32w + c is
  // kept in the rows of 128-row query tile qm (a broadcast dimension has coordinate 0)
  const uint32_t *blockmap;
  int bm_heads, bm_qtiles, bm_words;
  GQA_EXTENTS
};

// Whether the boolean mask keeps any key of [k0, k0 + 128) in this CTA's query tile for
// head h0 (or h0 + 1 when `two`): 8 bits of the block map from chunk k0 / 16.
__device__ __forceinline__ bool tile_kept(const PrefillArgs &a, int b, int h0, bool two, int qt, int k0) {
  const int c = k0 >> 4, w = c >> 5, sh = c & 31;
  const int bm = a.mask_bcast_b ? 0 : b, qm = a.mask_bcast_i ? 0 : qt;
  for (int hh = 0; hh < (two && !a.mask_bcast_h ? 2 : 1); ++hh) {
    const int hm = a.mask_bcast_h ? 0 : h0 + hh;
    const uint32_t *row = a.blockmap + (((size_t)bm * a.bm_heads + hm) * a.bm_qtiles + qm) * a.bm_words;
    uint64_t x = w < a.bm_words ? row[w] : 0u;
    if (w + 1 < a.bm_words) x |= (uint64_t)row[w + 1] << 32;
    if ((x >> sh) & 0xFFu) return true;
  }
  return false;
}


template <int D, int DV, int MK> struct PSmem {
  static constexpr int kTile = BM * D * 2;    // one Q or K tile
  static constexpr int kVTile = BN * DV * 2;  // one V tile
  static constexpr int kMaskTile = MK == 1 ? BM * BN : MK >= 2 ? BM * BN * 2 : 0;  // one buffer
  static constexpr int kMaskRing = MK == 3 ? 2 : 1;  // shared tiles in flight (MK 3)
  static constexpr int kMaskBufs = MK == 3 ? kMaskRing : 2;
  // the K ring gives up a stage when two would not leave room for the mask buffers
  static constexpr int kKStages =
      (4 * kTile + 2 * kVTile + kMaskBufs * kMaskTile + 2048 > 227 * 1024) ? 1 : 2;
  static constexpr int kQA = 0;
  static constexpr int kQB = kQA + kTile;
  static constexpr int kK = kQB + kTile;
  static constexpr int kV = kK + kKStages * kTile;  // two stages
  static constexpr int kM = kV + 2 * kVTile;        // mask tiles
  static constexpr int kBar = kM + kMaskBufs * kMaskTile;
  static constexpr int kTmemSlot = kBar + 24 * 8;
  static constexpr int kFlag = kTmemSlot + 8;
  // MK 1 with a block map: the count and the indices of the key tiles the mask keeps
  static constexpr int kMaxLive = 508;
  static constexpr int kLive = kFlag + 8;
  static constexpr int kBytes = kLive + 4 + kMaxLive * 2;
  // more than half of an SM's shared memory, so a CTA (512 TMEM columns) is always alone
  // on its SM and can never sit blocked in tcgen05.alloc behind another one
  static constexpr int kAlloc = (kBytes + 1024) > 116 * 1024 ? (kBytes + 1024) : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;  // S_A, S_B (128 each), O_A, O_B (128 each)
};

// Shared-memory matrix descriptor (tcgen05), 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for sm_10x
  d |= (uint64_t)2 << 61;  // 128B swizzle
  return d;
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
template <typename T> __host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn_major) {
  return (1u << 4)                                        // D format: f32
         | ((DT<T>::code == GQA_BF16 ? 1u : 0u) << 7)     // A format: bf16 / f16
         | ((DT<T>::code == GQA_BF16 ? 1u : 0u) << 10)    // B format
         | ((b_mn_major ? 1u : 0u) << 16)                 // B major-ness
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

#define GQA_REG32(r) \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),   \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),  \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : GQA_REG32(r)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Two additive mask values (one 32-bit word of the dtype) as a pair of floats.
template <typename T> __device__ __forceinline__ uint64_t bias_pair(uint32_t w);
template <> __device__ __forceinline__ uint64_t bias_pair<__nv_bfloat16>(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <> __device__ __forceinline__ uint64_t bias_pair<__half>(uint32_t w) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
  return f2_pack(f.x, f.y);
}

// Frontier tiles with a softcap: clear the packed P of the keys outside [lo_vis, hi_vis]
// in this lane's 64 TMEM columns of P and return how many there were.  Kept out of line so
// that the softmax loop around it compiles as without it.
__device__ __noinline__ int clear_masked_p(uint32_t tP, int k0, int lo_vis, int hi_vis) {
  int nm = 0;
  tmem_st_wait();
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint32_t pk[32];
    tmem_ld32(tP + half * 32, pk);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 64; ++e) {
      const int key = k0 + half * 64 + e;
      if (key < lo_vis || key > hi_vis) {
        pk[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
        ++nm;
      }
    }
    tmem_st32(tP + half * 32, pk);
  }
  return nm;
}

// mbarriers (indices into bars[])
enum {
  B_Q = 0,
  B_KFULL0, B_KFULL1, B_KEMPTY0, B_KEMPTY1,
  B_VFULL0, B_VFULL1, B_VEMPTY0, B_VEMPTY1,
  B_SFULL_A, B_SFULL_B, B_PFULL_A, B_PFULL_B, B_OFULL_A, B_OFULL_B,
  B_MFULL_A, B_MFULL_B, B_MEMPTY_A, B_MEMPTY_B,
  B_STALL,  // never completed (failure-path test hook)
  B_COUNT
};
static_assert(B_COUNT <= 24, "barrier region");

template <typename T, int D, int DV, bool SOFTCAP, int MK>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmm,
                      PrefillArgs a) {
  using L = PSmem<D, DV, MK>;
  constexpr int KST = L::kKStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kTmemSlot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kFlag);

  // CTA = (pair of q heads of one kv group, q tile, batch); longest q tiles first
  const int pairs_per_group = (a.G + 1) / 2;
  const int hk = blockIdx.x / pairs_per_group;
  const int hA = hk * a.G + 2 * (blockIdx.x % pairs_per_group);
  const bool has_b = hA + 1 < (hk + 1) * a.G;
  const int b = blockIdx.z;
  const int qt = gridDim.y - 1 - blockIdx.y;
  const int q0 = qt * BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int past = load_past(a.seqlens, a.nonpad, b, a.curr, a.cap);
  int st = sequence_status(past, a.curr, a.ring ? INT_MAX : a.cap, a.cap_past, a.past_separate, a.do_rotary,
                           a.rope_len);
  if (MK && !st && (long long)past + a.curr > a.mask_keys) st = GQA_DEV_BAD_SEQLEN;  // the mask must cover every key
  if (a.table && !st) {
    // every page of the sequence's band must exist: the same decision in every CTA of the
    // sequence and in the append kernel
    const int lo_seq = a.window > 0 ? max(0, past - a.window + 1) : 0, tot = past + a.curr;
    const int32_t *trow = a.table + (size_t)b * a.max_pages;
    bool bad = false;
    for (int n = lo_seq / 64 + (int)threadIdx.x; n * 64 < tot; n += blockDim.x)
      bad |= trow[n] < 0 || trow[n] >= a.num_pages;
    if (__syncthreads_or(bad)) st = GQA_DEV_BAD_PAGE;
  }
  T *out = reinterpret_cast<T *>(a.out);
  const int nrows = min(BM, a.curr - q0);
  if (st) {
    if (threadIdx.x == 0 && qt == 0 && blockIdx.x == 0) report(a.status, st);
    for (int idx = threadIdx.x; idx < (has_b ? 2 : 1) * nrows * DV; idx += blockDim.x) {
      const int hh = idx / (nrows * DV), r = (idx / DV) % nrows, d = idx % DV;
      GQA_GUARD((((size_t)b * a.curr + q0 + r) * a.Hq + hA + hh) * DV + d, 1, a.ext.out, a.status)
      out[(((size_t)b * a.curr + q0 + r) * a.Hq + hA + hh) * DV + d] = from_f32<T>(0.f);
    }
    return;
  }
  const int total = past + a.curr;
  const int qa_first = past + q0, qa_last = past + q0 + nrows - 1;
  int klo = a.window > 0 ? max(0, qa_first - a.window + 1) : 0;
  if (MK) klo &= ~15;  // the mask's TMA coordinate: a multiple of 16 bytes
  // a ring or paged cache: tiles start on 128-position boundaries, so a tile never straddles
  // the ring's wrap and is two whole pages; the extra keys fall outside the band (masked)
  if (a.ring || a.table) klo &= ~(BN - 1);
  const int khi = a.causal ? min(total, qa_last + 1) : total;
  const int ntiles_band = (khi - klo + BN - 1) / BN;  // >= 1: every row sees itself
  // boolean mask with a block map: only the tiles where the mask keeps a key of this query
  // tile are streamed, in order (every role walks the same list); otherwise every tile
  int *nlive = reinterpret_cast<int *>(smem + L::kLive);
  uint16_t *live = reinterpret_cast<uint16_t *>(smem + L::kLive + 4);
  const bool skip = MK == 1 && a.blockmap != nullptr && ntiles_band <= L::kMaxLive;
  if (skip && warp == 0) {
    int n = 0;
    for (int t0 = 0; t0 < ntiles_band; t0 += 32) {
      const int t = t0 + lane;
      const bool keep = t < ntiles_band && tile_kept(a, b, hA, has_b, qt, klo + t * BN);
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      if (keep) live[n + __popc(m & ((1u << lane) - 1u))] = (uint16_t)t;
      n += __popc(m);
    }
    if (lane == 0) *nlive = n;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(&bars[i], ((i == B_MEMPTY_A || i == B_MEMPTY_B) && MK == 3 && has_b) ? 8  // both heads read it
                          : (i == B_PFULL_A || i == B_PFULL_B || i == B_MEMPTY_A || i == B_MEMPTY_B) ? 4 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = skip ? *nlive : ntiles_band;  // tiles streamed
  // TMEM columns: S_A [0,128) S_B [128,256) O_A [256,256+DV) O_B [384,384+DV); P_X overwrites
  // the first 64 columns of S_X as packed pairs
  int kissued = 0, vissued = 0;      // producer thread: TMA tiles issued
  int missued[2] = {0, 0};           // mask producer thread: loads issued per buffer
  int s_commits = 0, o_commits = 0;  // MMA thread: last S and PV commit counts
  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      mbar_expect_tx(&bars[B_Q], (has_b ? 2 : 1) * L::kTile);
#pragma unroll
      for (int db = 0; db < D / 64; ++db) {
        tma_load_4d(smem + L::kQA + db * (BM * 128), &tmq, db * 64, hA, q0, b, &bars[B_Q]);
        if (has_b) tma_load_4d(smem + L::kQB + db * (BM * 128), &tmq, db * 64, hA + 1, q0, b, &bars[B_Q]);
      }
      const int bh = b * a.Hkv + hk;
      // (row, group) of the 64 keys from k0 in the K/V tensor maps: contiguous [B*Hkv][cap],
      // ring [B*Hkv][cap] at row k0 % cap, pool [num_pages*Hkv][64] at the page of k0.  Only
      // the pages of the sequence's band were checked: a 64-key half before the band's first
      // page or past its last key reads the nearest checked page instead (those keys are
      // never visible; rows past the last key have their V cleared before PV)
      const int32_t *trow = a.table ? a.table + (size_t)b * a.max_pages : nullptr;
      const int first_page = (a.window > 0 ? max(0, past - a.window + 1) : 0) / 64, last_page = (total - 1) / 64;
      auto half_coord = [&](int k0, int &row, int &group) {
        if (trow) {
          group = trow[min(max(k0 / 64, first_page), last_page)] * a.Hkv + hk;
          row = 0;
        } else {
          group = bh;
          row = a.ring ? k0 % a.cap : k0;
        }
      };
      // one 128-key tile of a K or V tensor map: a single box, or two 64-row boxes of pages
      auto load_tile = [&](uint8_t *dst, const CUtensorMap *map, int k0, int cols, uint64_t *bar) {
#pragma unroll 1
        for (int db = 0; db < cols / 64; ++db) {
          int row, group;
          half_coord(k0, row, group);
          tma_load_3d(dst + db * (BN * 128), map, db * 64, row, group, bar);
          if (trow) {
            half_coord(k0 + 64, row, group);
            tma_load_3d(dst + db * (BN * 128) + 64 * 128, map, db * 64, row, group, bar);
          }
        }
      };
      for (int t = 0; t < ntiles; ++t) {
        const int s = t & 1, k0 = klo + (skip ? live[t] : t) * BN, sk = t % KST;
        if (t >= KST && !mbar_wait(&bars[B_KEMPTY0 + sk], ((t / KST) - 1) & 1, abort_flag, a.wait_limit)) break;
        mbar_expect_tx(&bars[B_KFULL0 + sk], L::kTile);
        load_tile(smem + L::kK + sk * L::kTile, &tmk, k0, D, &bars[B_KFULL0 + sk]);
        ++kissued;
        if (t >= 2 && !mbar_wait(&bars[B_VEMPTY0 + s], ((t >> 1) - 1) & 1, abort_flag, a.wait_limit)) break;
        mbar_expect_tx(&bars[B_VFULL0 + s], L::kVTile);
        load_tile(smem + L::kV + s * L::kVTile, &tmv, k0, DV, &bars[B_VFULL0 + s]);
        ++vissued;
      }
    }
  } else if (MK && warp == 2) {
    // ---------------------------------------------------------------- mask producer
    if (lane == 0) {
      tma_prefetch_desc(&tmm);
      const int mrows = a.mask_bcast_i ? 1 : BM;
      const uint32_t bytes = (uint32_t)mrows * 128u * (MK >= 2 ? 2u : 1u);
      const int mb = a.mask_bcast_b ? 0 : b, mq = a.mask_bcast_i ? 0 : q0;
      for (int t = 0; t < ntiles; ++t) {
        const int k0 = klo + (skip ? live[t] : t) * BN;
        bool fine = true;
        // MK 1, 2: one buffer per head; MK 3: the shared tile goes to ring slot t % kMaskRing
        for (int h = 0; h < (MK != 3 && has_b ? 2 : 1); ++h) {
          const int slot = MK == 3 ? t % L::kMaskRing : h, use = MK == 3 ? t / L::kMaskRing : t;
          if (use >= 1 && !mbar_wait(&bars[B_MEMPTY_A + slot], (use - 1) & 1, abort_flag, a.wait_limit)) {
            fine = false;
            break;
          }
          const int mh = a.mask_bcast_h ? 0 : hA + h;
          uint8_t *dst = smem + L::kM + slot * L::kMaskTile;
          mbar_expect_tx(&bars[B_MFULL_A + slot], bytes);
          tma_load_4d(dst, &tmm, k0, mq, mh, mb, &bars[B_MFULL_A + slot]);
          if (MK >= 2) tma_load_4d(dst + BM * 128, &tmm, k0 + 64, mq, mh, mb, &bars[B_MFULL_A + slot]);
          missued[slot] = use + 1;
        }
        if (!fine) break;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t qa = smem_u32(smem + L::kQA), qb = smem_u32(smem + L::kQB);
    const uint32_t kbase = smem_u32(smem + L::kK), vbase = smem_u32(smem + L::kV);
    constexpr uint32_t id_s = idesc<T>(BM, BN, false);
    constexpr uint32_t id_pv = idesc<T>(BM, DV, true);
    auto issue_s = [&](int t, uint32_t q_s, uint32_t d_tmem) {
      const uint32_t ks = kbase + (t % KST) * L::kTile;
#pragma unroll
      for (int k16 = 0; k16 < D / 16; ++k16) {
        const uint32_t off = (k16 >> 2) * (BM * 128) + (k16 & 3) * 32;
        mma_ss(d_tmem, sdesc(q_s + off, 16, 1024), sdesc(ks + off, 16, 1024), id_s, k16 > 0);
      }
    };
    auto issue_pv = [&](int t, uint32_t p_tmem, uint32_t o_tmem) {
      const uint32_t vs = vbase + (t & 1) * L::kVTile;
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)
        mma_ts(o_tmem, p_tmem + kk * 8, sdesc(vs + kk * 2048, BN * 128, 1024), id_pv, (t > 0 || kk > 0) ? 1u : 0u);
    };
    // failure-path test hook: first a wait that nothing completes
    bool ok = !(a.stall && !__all_sync(0xffffffffu, mbar_wait(&bars[B_STALL], 0, abort_flag, a.wait_limit))) &&
              __all_sync(0xffffffffu, mbar_wait(&bars[B_Q], 0, abort_flag, a.wait_limit)) && (MK != 1 || ntiles > 0) &&
              __all_sync(0xffffffffu, mbar_wait(&bars[B_KFULL0], 0, abort_flag, a.wait_limit));
    if (ok) {
      tc_fence_after();
      if (lane == 0) {
        issue_s(0, qa, tmem + 0);
        tc_commit(&bars[B_SFULL_A]);
        if (has_b) {
          issue_s(0, qb, tmem + 128);
          tc_commit(&bars[B_SFULL_B]);
        }
        tc_commit(&bars[B_KEMPTY0]);
      }
      s_commits = 1;
      __syncwarp();
    }
    for (int t = 0; ok && t < ntiles; ++t) {
      const int s = t & 1, k0 = klo + (skip ? live[t] : t) * BN;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_VFULL0 + s], (t >> 1) & 1, abort_flag, a.wait_limit))) break;
      if (k0 + BN > total) {  // stale slots may hold NaN/Inf: zero those V rows
        const int first = max(0, total - k0);
        uint8_t *vb = smem + L::kV + s * L::kVTile;
        for (int idx = lane; idx < (BN - first) * (DV / 8); idx += 32) {
          const int r = first + idx / (DV / 8), ch = idx % (DV / 8);
          *reinterpret_cast<uint4 *>(vb + (ch >> 3) * (BN * 128) + sw128(r, ch & 7)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_PFULL_A], t & 1, abort_flag, a.wait_limit))) break;
      tc_fence_after();
      if (lane == 0) {
        issue_pv(t, tmem + 0, tmem + 256);
        tc_commit(&bars[B_OFULL_A]);
      }
      __syncwarp();
      const bool next = t + 1 < ntiles;
      if (next) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bars[B_KFULL0 + (t + 1) % KST], ((t + 1) / KST) & 1, abort_flag, a.wait_limit)))
          break;
        tc_fence_after();
        if (lane == 0) {
          issue_s(t + 1, qa, tmem + 0);
          tc_commit(&bars[B_SFULL_A]);
        }
        __syncwarp();
      }
      if (has_b) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_PFULL_B], t & 1, abort_flag, a.wait_limit))) break;
        tc_fence_after();
        if (lane == 0) {
          issue_pv(t, tmem + 128, tmem + 384);
          tc_commit(&bars[B_OFULL_B]);
        }
        __syncwarp();
      }
      if (lane == 0) tc_commit(&bars[B_VEMPTY0 + s]);
      o_commits = t + 1;
      if (next) {
        if (lane == 0) {
          if (has_b) {
            issue_s(t + 1, qb, tmem + 128);
            tc_commit(&bars[B_SFULL_B]);
          }
          tc_commit(&bars[B_KEMPTY0 + (t + 1) % KST]);
        }
        s_commits = t + 2;
        __syncwarp();
      }
    }
  } else if (warp >= 4 && (warp < 8 || has_b)) {
    // ---------------------------------------------------------------- softmax warpgroups
    const int wg = (warp - 4) >> 2;  // 0: head A, 1: head B
    const int hq = hA + wg;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // TMEM lane = query row within the tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + wg * 128;
    const uint32_t tO = tmem + lane_off + 256 + wg * 128;
    uint64_t *sfull = &bars[B_SFULL_A + wg], *pfull = &bars[B_PFULL_A + wg], *ofull = &bars[B_OFULL_A + wg];
    const int qa = past + q0 + row;
    const float z2 = a.has_sink ? (a.head_sink ? a.head_sink[hq] : 0.f) * kLog2e : 0.f;
    const float smul = a.score_mul, cmul = a.cap_mul;
    float m_ref = a.has_sink ? z2 : -INFINITY;  // reference max (log2 domain)
    float l = a.has_sink ? 1.f : 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int k0 = klo + (skip ? live[t] : t) * BN;
      const bool edge = !(k0 + BN - 1 < total && (!a.causal || k0 + BN - 1 <= qa_first) &&
                          (a.window < 0 || qa_last - k0 < a.window));
      if (!__all_sync(0xffffffffu, mbar_wait(sfull, t & 1, abort_flag, a.wait_limit))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[BN];
      {
        uint32_t(&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
        uint32_t(&r1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
        uint32_t(&r2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[64]);
        uint32_t(&r3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[96]);
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_ld_wait();
      }
      if constexpr (MK != 0) {
        // this row's mask values for keys [k0, k0 + 128), 16-byte chunks of the 128B-swizzled
        // tile (row-broadcast masks hold one row)
        const int mbuf = MK == 3 ? t % L::kMaskRing : wg, muse = MK == 3 ? t / L::kMaskRing : t;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_MFULL_A + mbuf], muse & 1, abort_flag, a.wait_limit))) {
          ok = false;
          break;
        }
        const int mr = a.mask_bcast_i ? 0 : row;
        const uint8_t *mrow = smem + L::kM + mbuf * L::kMaskTile + mr * 128;
        if constexpr (MK == 1) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = *reinterpret_cast<const uint4 *>(mrow + ((ch ^ (mr & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (((w[e >> 2] >> (8 * (e & 3))) & 0xFFu) == 0u) r[ch * 16 + e] = __float_as_uint(-INFINITY);
          }
        } else {
          // r += bias / scale, two keys per instruction (an additive -inf makes r -inf: weight
          // 0 without a softcap, the score -softcap through tanh with one)
          const uint64_t bm2 = f2_pack(a.bias_mul, a.bias_mul);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint4 v = *reinterpret_cast<const uint4 *>(mrow + hf * (BM * 128) + ((ch ^ (mr & 7)) << 4));
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                uint32_t &r0 = r[hf * 64 + ch * 8 + e], &r1 = r[hf * 64 + ch * 8 + e + 1];
                const float2 y = f2_unpack(f2_fma(bias_pair<T>(w[e >> 1]), bm2, f2_pack(__uint_as_float(r0),
                                                                                         __uint_as_float(r1))));
                r0 = __float_as_uint(y.x);
                r1 = __float_as_uint(y.y);
              }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_MEMPTY_A + mbuf]);
      }
      if (edge) {  // band predicate on frontier tiles only
        const int lo_vis = a.window > 0 ? qa - a.window + 1 : INT_MIN;
        const int hi_vis = a.causal ? min(qa, total - 1) : total - 1;
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          const int key = k0 + e;
          if (key < lo_vis || key > hi_vis) r[e] = __float_as_uint(-INFINITY);
        }
      }
      // row maximum over four independent chains (a single chain of 64 dependent steps was
      // a measured latency bottleneck), combined at the end
      float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < BN; e += 2)
        mxs[(e >> 1) & 3] = fmax3(mxs[(e >> 1) & 3], __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
      float mx = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3]));
      // under a softcap an additive -inf still scores -softcap: the maximum counts it
      if (MK >= 2 && SOFTCAP) mx = fmaxf(mx, -FLT_MAX);
      float m_tile = -INFINITY;
      if (mx != -INFINITY) m_tile = SOFTCAP ? tanh_fast(mx * smul) * cmul : mx * smul;
      // lazy rescale: move the reference max only when it grows by more than 2^8
      const bool need = m_tile > m_ref + kRescaleLog2 || (m_ref == -INFINITY && m_tile != -INFINITY);
      const float m_new = need ? m_tile : m_ref;
      const float alpha = need ? ex2(m_ref - m_new) : 1.f;
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      // P = 2^(x - m) in two halves (keeps register pressure down), packed to the dtype and
      // stored over the first columns of S; elementwise math two lanes per instruction
      uint64_t rs2[2] = {0, 0};  // (0.f, 0.f): two independent row-sum chains
      const uint64_t smul2 = f2_pack(smul, smul), cmul2 = f2_pack(cmul, cmul), negm2 = f2_pack(-m_use, -m_use);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const uint64_t sv = f2_pack(__uint_as_float(r[half * 64 + e]), __uint_as_float(r[half * 64 + e + 1]));
          uint64_t x;
          if (SOFTCAP) {
            const float2 y = f2_unpack(f2_mul(sv, smul2));
            x = f2_fma(f2_pack(tanh_fast(y.x), tanh_fast(y.y)), cmul2, negm2);
          } else {
            x = f2_fma(sv, smul2, negm2);
          }
          const float2 xf = f2_unpack(x);
          float p0 = ex2(xf.x), p1 = ex2(xf.y);
          if (MK == 1 && SOFTCAP) {  // removed keys (band or mask) have weight exactly zero
            if (r[half * 64 + e] == __float_as_uint(-INFINITY)) p0 = 0.f;
            if (r[half * 64 + e + 1] == __float_as_uint(-INFINITY)) p1 = 0.f;
          }
          rs2[(e >> 1) & 1] = f2_add(rs2[(e >> 1) & 1], f2_pack(p0, p1));
          pk[e >> 1] = pack2<T>(p0, p1);
        }
        tmem_st32(tS + half * 32, pk);
      }
      const float2 rsf = f2_unpack(f2_add(rs2[0], rs2[1]));
      float rs = rsf.x + rsf.y;
      if (MK != 1 && SOFTCAP && edge) {
        // a masked key's -inf came out of tanh as -1, i.e. a score of -softcap: clear its P
        // (the same value for every masked key of the row) in TMEM and take it out of the
        // row sum, so that a masked key has exactly zero weight.  Frontier tiles only.
        const int lo_vis = a.window > 0 ? qa - a.window + 1 : INT_MIN;
        const int hi_vis = a.causal ? min(qa, total - 1) : total - 1;
        const float pm = ex2(fmaf(-1.f, cmul, -m_use));
        rs -= (float)clear_masked_p(tS, k0, lo_vis, hi_vis) * pm;
      }
      l = l * alpha + rs;
      m_ref = m_new;
      if (__any_sync(0xffffffffu, need) && t > 0) {
        // O holds PV of tiles < t: wait for the last of them, then scale it in TMEM
        if (!__all_sync(0xffffffffu, mbar_wait(ofull, (t - 1) & 1, abort_flag, a.wait_limit))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull);
    }
    // epilogue: out = O / l
    const bool none = MK == 1 && ntiles == 0;  // the mask keeps no key of this query tile
    const bool fin = ok && !*abort_flag && (none || mbar_wait(ofull, (ntiles - 1) & 1, abort_flag, a.wait_limit));
    if (__all_sync(0xffffffffu, fin) && none) {
      T *orow = out + (((size_t)b * a.curr + q0 + row) * a.Hq + hq) * DV;
      if (row < nrows)
        for (int c = 0; c < DV; c += 8) {
          GQA_GUARD((((size_t)b * a.curr + q0 + row) * a.Hq + hq) * DV + c, 8, a.ext.out, a.status)
          *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0, 0, 0, 0);
        }
    } else if (__all_sync(0xffffffffu, fin)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      T *orow = out + (((size_t)b * a.curr + q0 + row) * a.Hq + hq) * DV;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait();
        if (row < nrows) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v;
            v.x = pack2<T>(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
            v.y = pack2<T>(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            v.z = pack2<T>(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
            v.w = pack2<T>(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
            GQA_GUARD((((size_t)b * a.curr + q0 + row) * a.Hq + hq) * DV + c * 32 + e, 8, a.ext.out, a.status)
            *reinterpret_cast<uint4 *>(orow + c * 32 + e) = v;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait timed out somewhere.  Copies and MMAs already issued must land before the
    // CTA exits and before its TMEM is freed; these waits are bounded too.
    volatile int no_abort = 0;
    if (warp == 0 && lane == 0) {
      mbar_wait(&bars[B_Q], 0, &no_abort);
      for (int t = max(0, kissued - KST); t < kissued; ++t)
        mbar_wait(&bars[B_KFULL0 + t % KST], (t / KST) & 1, &no_abort);
      for (int t = max(0, vissued - 2); t < vissued; ++t) mbar_wait(&bars[B_VFULL0 + (t & 1)], (t >> 1) & 1, &no_abort);
      report(a.status, GQA_DEV_TIMEOUT);
    }
    if (MK && warp == 2 && lane == 0) {
      for (int h = 0; h < 2; ++h)
        if (missued[h]) mbar_wait(&bars[B_MFULL_A + h], (missued[h] - 1) & 1, &no_abort);
    }
    if (warp == 1 && lane == 0) {
      if (s_commits) mbar_wait(&bars[B_SFULL_A], (s_commits - 1) & 1, &no_abort);
      if (o_commits) mbar_wait(&bars[B_OFULL_A], (o_commits - 1) & 1, &no_abort);
      if (has_b && o_commits) mbar_wait(&bars[B_OFULL_B], (o_commits - 1) & 1, &no_abort);
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <typename T, int D, int DV, bool SC, int MK> gqa_status launch_cfg(const Call &c, const PrefillArgs &a) {
  using L = PSmem<D, DV, MK>;
  static_assert(L::kAlloc <= 227 * 1024, "shared memory per CTA");
  const gqa_params &p = c.p;
  CUtensorMap tq, tk, tv, tm;
  const bool paged = c.block_table != nullptr;
  const long long outer = paged ? (long long)c.num_pages * p.kv_heads : (long long)p.batch * p.kv_heads;
  const int rows = paged ? 64 : p.cap_present, box_rows = paged ? 64 : BN;
  if (!encode_q_map(&tq, c.q, D, p.q_heads, p.q_len, p.batch, BM, 2)) return GQA_ERR_CUDA;
  if (!encode_kv_map(&tk, c.present_k, D, rows, outer, box_rows, 2)) return GQA_ERR_CUDA;
  if (!encode_kv_map(&tv, c.present_v, DV, rows, outer, box_rows, 2)) return GQA_ERR_CUDA;
  if (MK) {
    const int es = MK >= 2 ? 2 : 1;
    if (!encode_mask_map(&tm, c.mask, c.mask_keys, p.q_len, p.q_heads, p.batch, c.mask_si * es, c.mask_sh * es,
                         c.mask_sb * es, 128 / es, c.mask_si == 0 ? 1 : BM, es))
      return GQA_ERR_CUDA;
  } else {
    tm = tq;  // unused
  }
  auto kern = prefill_tc_kernel<T, D, DV, SC, MK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess)
    return GQA_ERR_CUDA;
  const int pairs = p.kv_heads * ((c.G + 1) / 2);
  dim3 grid(pairs, (p.q_len + BM - 1) / BM, p.batch);
  kern<<<grid, kThreads, L::kAlloc, c.stream>>>(tq, tk, tv, tm, a);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

template <typename T, int MK, bool MIXED> gqa_status launch_t(const Call &c) {
  const gqa_params &p = c.p;
  PrefillArgs a;
  a.out = c.out;
  a.seqlens = c.seqlens;
  a.nonpad = c.nonpad;
  a.head_sink = c.head_sink;
  a.status = c.status;
  a.Hq = p.q_heads;
  a.Hkv = p.kv_heads;
  a.G = c.G;
  a.curr = p.q_len;
  a.cap = p.cap_present;
  a.cap_past = p.cap_past;
  a.past_separate = c.past_separate;
  a.rope_len = p.rope_len;
  a.do_rotary = c.append ? p.do_rotary : 0;
  a.window = p.window;
  a.causal = p.causal;
  a.has_sink = (c.head_sink != nullptr) || p.smooth_softmax;
  a.mask_keys = c.mask_keys;
  a.mask_bcast_b = c.mask_sb == 0;
  a.mask_bcast_h = c.mask_sh == 0;
  a.mask_bcast_i = c.mask_si == 0;
  a.bias_mul = 1.f / p.scale;
  a.wait_limit = c.wait_limit > 0 ? c.wait_limit : kWaitLimitCycles;
  a.stall = c.stall;
  a.ring = p.kv_ring;
  a.table = c.block_table;
  a.max_pages = c.max_pages;
  a.num_pages = c.num_pages;
  a.blockmap = MK == 1 ? c.blockmap : nullptr;
  a.bm_heads = c.mask_sh == 0 ? 1 : p.q_heads;
  a.bm_qtiles = c.mask_si == 0 ? 1 : (p.q_len + BM - 1) / BM;
  a.bm_words = (((c.mask_keys < p.cap_present ? c.mask_keys : p.cap_present) + 15) / 16 + 31) / 32;
#ifdef GQA_BOUNDS_CHECK
  a.ext = extents_of(c, WsLayout{});
#endif
  const bool sc = p.softcap > 0.f;
  if (sc) {
    a.score_mul = p.scale / p.softcap;
    a.cap_mul = p.softcap * kLog2e;
  } else {
    a.score_mul = p.scale * kLog2e;
    a.cap_mul = 0.f;
  }
  const int D = p.head_dim, DV = c.Dv;
  if constexpr (!MIXED) {
    if (D == 128 && DV == 128) return sc ? launch_cfg<T, 128, 128, true, MK>(c, a) : launch_cfg<T, 128, 128, false, MK>(c, a);
    if (D == 64 && DV == 64) return sc ? launch_cfg<T, 64, 64, true, MK>(c, a) : launch_cfg<T, 64, 64, false, MK>(c, a);
  } else {  // V head dim != Q/K head dim
    if (D == 128 && DV == 64) return sc ? launch_cfg<T, 128, 64, true, MK>(c, a) : launch_cfg<T, 128, 64, false, MK>(c, a);
    if (D == 64 && DV == 128) return sc ? launch_cfg<T, 64, 128, true, MK>(c, a) : launch_cfg<T, 64, 128, false, MK>(c, a);
  }
  return GQA_ERR_UNSUPPORTED;
}

// one dtype switch per (MK, MIXED); each .cu file instantiates its own set
template <int MK, bool MIXED> gqa_status launch_prefill_tc_any(const Call &c) {
  switch (c.p.dtype) {
    case GQA_F16: return launch_t<__half, MK, MIXED>(c);
    case GQA_BF16: return launch_t<__nv_bfloat16, MK, MIXED>(c);
  }
  return GQA_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace gqa

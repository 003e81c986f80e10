// common.cuh -- device helpers shared by the kernels of libgqa: inline PTX for mbarriers,
// TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, ld/st, commit), ldmatrix and
// mma.sync, plus bounded waits.  Written from the PTX ISA's instruction descriptions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gqa.h"

namespace gqa {

// A pipeline wait that has not completed after this many SM cycles (about 2 s at the
// GB300's 2.07 GHz maximum SM clock, up to 4 s at 1 GHz) gives up, sets GQA_DEV_TIMEOUT
// and lets the kernel drain and return instead of hanging the GPU.  The SM cycle counter is cheap to read, unlike the global
// timer, so the bound costs nothing on the fast path.
constexpr long long kWaitLimitCycles = 4000000000ll;

constexpr float kLog2e = 1.4426950408889634f;

template <typename T> struct DT;
template <> struct DT<float> { static constexpr int code = GQA_F32; };
template <> struct DT<__half> { static constexpr int code = GQA_F16; };
template <> struct DT<__nv_bfloat16> { static constexpr int code = GQA_BF16; };

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// f8 E4M3 codes of a quantized KV cache, through the hardware conversions.  Both 8-bit
// halves of the pair carry the same value, so the result does not depend on which half an
// instruction reads or writes.  To a code: nearest, ties to even, saturating at +-448
// (infinity too), NaN to NaN.  From a code: exact (every E4M3 value is an f16 value).
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(x));
  return (uint8_t)(r & 0xFFu);
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  const uint32_t h = e4m3x2_to_f16x2((uint16_t)(c | (c << 8)));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// int8 codes of a quantized KV cache: to a code, round half to even and saturate at -128
// and 127 (infinities too), NaN to 0; from a code, exact.  The pair conversion biases each
// code by 128 (its sign bit flipped) and places it in the low byte of an f16 whose high
// byte is 0x64, i.e. 1024 + code + 128, then subtracts 1152 (0x6480): both steps are exact.
__device__ __forceinline__ uint8_t f32_to_s8(float x) {
  int r;
  asm("cvt.rni.sat.s32.f32 %0, %1;" : "=r"(r) : "f"(x));
  r = min(max(r, -128), 127);
  return isnan(x) ? (uint8_t)0 : (uint8_t)(r & 0xFF);
}
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint16_t codes) {
  const uint32_t w = __byte_perm((uint32_t)codes ^ 0x8080u, 0x64646464u, 0x5140);
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0x64806480u));
  return r;
}
__device__ __forceinline__ float s8_to_f32(uint8_t c) { return (float)(int8_t)c; }

// one-byte cache codes: E4M3, or int8 when I8
template <bool I8> __device__ __forceinline__ uint8_t f32_to_code(float x) {
  if constexpr (I8) return f32_to_s8(x);
  else return f32_to_e4m3(x);
}
template <bool I8> __device__ __forceinline__ uint32_t codes2_to_f16x2(uint16_t codes) {
  if constexpr (I8) return s8x2_to_f16x2(codes);
  else return e4m3x2_to_f16x2(codes);
}
// The four codes of w as two f16x2 words: PAIRS 0 takes bytes (0, 1) into lo and (2, 3)
// into hi; PAIRS 1 takes bytes (0, 2) into lo and (1, 3) into hi (lower byte, lower half).
// int8: one bias for the four codes, then one byte permute and one subtraction per pair.
template <bool I8, int PAIRS>
__device__ __forceinline__ void codes4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  if constexpr (I8) {
    const uint32_t x = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(x, 0x64646464u, PAIRS ? 0x4240 : 0x4140);
    const uint32_t b = __byte_perm(x, 0x64646464u, PAIRS ? 0x4341 : 0x4342);
    asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
  } else {
    const uint32_t x = PAIRS ? __byte_perm(w, 0, 0x3120) : w;
    lo = e4m3x2_to_f16x2((uint16_t)(x & 0xFFFFu));
    hi = e4m3x2_to_f16x2((uint16_t)(x >> 16));
  }
}
template <bool I8> __device__ __forceinline__ float code_to_f32(uint8_t c) {
  if constexpr (I8) return s8_to_f32(c);
  else return e4m3_to_f32(c);
}

// Per-sequence validity shared by every kernel: the same rule decides what is appended
// and which outputs are zeroed.  Returns GQA_DEV_* bits (0 = valid).
__device__ __forceinline__ int sequence_status(int past, int curr, int cap_present, int cap_past,
                                               int past_separate, int do_rotary, int rope_len) {
  if (past < 0 || (long long)past + curr > cap_present || (past_separate && past > cap_past))
    return GQA_DEV_BAD_SEQLEN;
  if (do_rotary && (long long)past + curr > rope_len) return GQA_DEV_BAD_ROPE_POS;
  return 0;
}

// The past length of sequence b: seqlens_k[b], or, for a padded cache (nonpad != NULL, the
// opset-24 nonpad_kv_seqlen: n valid keys, the curr queries the last curr of them),
// n - curr; an n outside [curr, cap] gives -1, which sequence_status rejects.
__device__ __forceinline__ int load_past(const int32_t *seqlens, const int64_t *nonpad, int b, int curr, int cap) {
  if (!nonpad) return seqlens[b];
  const long long n = nonpad[b];
  return (n >= curr && n <= cap) ? (int)(n - curr) : -1;
}

__device__ __forceinline__ void report(int32_t *status, int bits) {
  if (status && bits) atomicOr(status, bits);
}

// Bounds-checked debug build (-DGQA_BOUNDS_CHECK; the stand-in for a memory checker): every
// global store of the kernels is preceded by GQA_GUARD(first element, elements, the buffer's
// extent in elements, status), which skips a store that would leave its buffer and sets
// GQA_DEV_BOUNDS.  The extents come from the call (Extents, filled on the host).  In the
// product build the guard expands to nothing.
#ifdef GQA_BOUNDS_CHECK
constexpr int kDevBounds = 16;
__device__ __forceinline__ bool store_ok(size_t off, size_t n, size_t extent, int32_t *status) {
  if (off + n <= extent) return true;
  report(status, kDevBounds);
  return false;
}
#define GQA_GUARD(off, n, extent, status) \
  if (::gqa::store_ok((size_t)(off), (size_t)(n), (size_t)(extent), (status)))
#define GQA_EXTENTS Extents ext;
#define GQA_EXT(field) a.ext.field
#else
#define GQA_EXT(field) ((size_t)0)
#define GQA_GUARD(off, n, extent, status)
#define GQA_EXTENTS
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ packed fp32 (sm_100+)
// Two fp32 lanes per instruction: halves the issue slots of elementwise softmax math.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up (returns false) when
// *abort is set by another thread or when `limit` SM cycles have passed, in which case it
// sets *abort itself so that every role of the CTA winds down.  Pipeline waits pass the
// launch's limit (kWaitLimitCycles unless a test shortened it); the waits that drain copies
// and MMAs already in flight keep the full bound.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > limit) {
        *abort = 1;
        return false;
      }
    }
  }
}

// As mbar_wait, for a phase completed by other CTAs of the cluster: acquire at cluster scope,
// so their stores are visible once it returns true.  Bounded by kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 15u) == 15u && clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
// 16-byte asynchronous copy global -> shared (completion tracked per thread by cp.async groups).
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Generic-proxy writes to shared memory made visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ named barriers
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier among `nthreads` threads that also returns the OR of `pred` over them, so that a
// decision taken after it is the same for every participating thread.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ thread-block clusters
// Barrier over every thread of every CTA of the cluster; release/acquire order shared-memory
// writes before it with distributed shared-memory reads after it.  Every CTA of the cluster
// must reach it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split form of cluster_sync: arrive early, do other work, then wait.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
// Arrival that orders no memory access: only "this CTA got here" is signalled.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Stores into another CTA's shared memory (address from cluster_map); visible to it after
// the next cluster barrier.
__device__ __forceinline__ void cluster_st(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Stores into another CTA's shared memory that complete a transaction count on an mbarrier
// of that CTA (both addresses from cluster_map): the receiver waits on its own barrier
// instead of a cluster-wide one.
__device__ __forceinline__ void cluster_st_async4(uint32_t addr, float4 v, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void cluster_st_async2(uint32_t addr, float x, float y, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(x), "f"(y), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void cluster_st4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// ------------------------------------------------------------------ ldmatrix / mma.sync
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// transpose of an 8x8 matrix of 16-bit values held one row-pair per lane (the ldmatrix
// fragment layout: lane i has row i/4, columns 2(i%4) and 2(i%4) + 1)
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <typename T> struct Mma16816;
template <> struct Mma16816<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};
template <> struct Mma16816<__half> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a 128-byte-swizzled tile:
// rows are 128 bytes, and chunk c of row r is stored at chunk c ^ (r % 8).  This is the
// layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B and that tcgen05 descriptors with
// the 128B swizzle mode read (tile base aligned to 1024 bytes).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace gqa

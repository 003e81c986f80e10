/*
 * gqa.h -- C ABI of the sliding-window grouped-query attention library (libgqa.so).
 *
 * The library computes grouped-query attention (GQA) over a KV cache with the semantics
 * of com.microsoft.GroupQueryAttention / ONNX Attention, on one NVIDIA GB300 (sm_103a).
 * Every step runs in the library's own CUDA kernels; nothing falls back to the CPU.
 *
 * Passages that define the operation (cited by page title and section):
 *  [P1] OpenVINO PR #37423 "[NPUW] Support GQA sliding-window and smooth-softmax in
 *       DecomposeGQA": "Sliding window" (mask key k_abs for query q_abs when
 *       q_abs - k_abs >= local_window_size, in true absolute positions; multi-token
 *       decode), "smooth_softmax / head_sink" (a per-head sink logit that joins the
 *       softmax denominator and is then dropped; zero sink for plain smooth_softmax).
 *  [P2] tract PR #2645 "onnx: import GroupQueryAttention decode steps and its internal
 *       rotary": "What changed" (past_key/past_value concatenated with the step into
 *       present_key/present_value; bottom-right causal band; do_rotary with positions
 *       0..S-1 for a first prompt and seqlens_k onward for generated tokens; K rotated
 *       before it enters the cache; causal=0 honoured).
 *  [P3] ExecuTorch PR #21901 "Add sliding windows to the off-graph KV-cache reference":
 *       the window is a per-layer setting and masks the cache rather than evicting it.
 *  [P4] onnx-light-cpu "Attention Kernel Design": "Layouts and semantics" (rank-3
 *       [B, L, H*D] tensors; group_size = q_heads / kv_heads maps q heads onto kv heads
 *       without repeating K or V; softcap; a V head dimension that may differ from the
 *       Q/K one), "Compute paths" (streaming online softmax,
 *       frontier block skipping), "Scheduling, precision, and invariants" (fp32
 *       accumulation, output narrowed once; invalid combinations fail explicitly; a fully
 *       masked row yields zeros, not NaN).
 *
 * Notation: B batch, Hq q heads, Hkv kv heads, G = Hq / Hkv, D head dim of q and k, Dv
 * head dim of v and out (v_head_dim, D when 0), curr = q_len new tokens per sequence,
 * past_b = seqlens_k[b], total_b = past_b + curr, cap = capacity.
 *
 * Layouts (all row-major, dense, no padding):
 *   q, q_rot        [B, curr, Hq*D]       element type = dtype
 *   out             [B, curr, Hq*Dv]
 *   k               [B, curr, Hkv*D]      new keys of this step
 *   v               [B, curr, Hkv*Dv]     new values of this step
 *   past_k          [B, Hkv, cap_past, D]       past_v  [B, Hkv, cap_past, Dv]
 *   present_k       [B, Hkv, cap_present, D]    present_v [B, Hkv, cap_present, Dv]
 *                   slot j holds absolute position j
 *   cos/sin_cache   [rope_len, D/2]       dtype; rotation of half-split pairs (d, d+D/2)
 *   seqlens_k       int32 [B] on the device (a [B,1] tensor works too) = valid past tokens
 *   head_sink       fp32 [Hq] on the device, or NULL
 *
 * Semantics of one call, per sequence b, q head h, new token i (q_abs = past_b + i):
 *   present[b, h/G, past_b + i] = rope(k[b, i, h/G], pos = past_b + i)   (rope only when
 *   do_rotary), present_v likewise without rope; q is rotated the same way.
 *   Slot j is visible iff j < total_b, (causal == 0 or j <= q_abs), and
 *   (window < 0 or q_abs - j < window).
 *   s_j = scale * <q_rot, k_j>; if softcap > 0, s_j = softcap * tanh(s_j / softcap).
 *   out = sum_j e^{s_j - M} v_j / (sink_term + sum_j e^{s_j - M}), M the row max, where
 *   sink_term = e^{z - M} with z = head_sink[h] (or z = 0 if smooth_softmax and head_sink
 *   is NULL), else 0.  The sink is neither scaled nor capped.  A row with no visible slot
 *   gives zeros.
 *
 * Ring cache (kv_ring = 1; [P1] "Sliding window": sliding_window_cache, the rolling KV
 * buffer whose memory is bounded by the window): present holds cap_present slots and
 * absolute position p lives in slot p mod cap_present, so a layer with window W needs
 * only W + curr - 1 slots whatever the sequence length.  Requires window >= 1 and
 * window + q_len - 1 <= cap_present (else GQA_ERR_CAPACITY: a key the step sees would
 * already be overwritten), cap_present a multiple of 64 (else GQA_ERR_UNSUPPORTED),
 * present aliasing past (the ring is updated in place; else GQA_ERR_INVALID_ARG), and either
 * the decode entry points on the split-KV kernel's shapes (bf16/f16), or
 * gqa_attention_prefill (a prompt, or a chunk of one, appended into the ring; bf16/f16 and
 * cap_present a multiple of 128, since the tensor-core prefill reads 128-position tiles);
 * other combinations return GQA_ERR_UNSUPPORTED.  seqlens_k is the absolute past length and
 * may exceed cap_present; the band predicate is unchanged.  gqa_rope_append_kv appends into
 * a ring the same way.
 *
 * Ownership and memory: the caller owns every buffer; all pointers except the params and
 * mask structs are device pointers, 16-byte aligned (seqlens_k, head_sink and the f8
 * scales 4-byte aligned).  The library allocates no memory (it uses
 * the caller's workspace) and keeps no state between calls apart from the counters it
 * leaves zeroed in the workspace.  present may alias past (same pointer): an in-place
 * append that writes only rows [past_b, total_b).  Otherwise rows [0, past_b) of past are
 * copied into present first; partially overlapping buffers are not allowed.  Rows of
 * present at or beyond total_b are neither read nor written.
 *
 * Streams and errors: every call enqueues its kernels on `stream` (a cudaStream_t, NULL
 * for the legacy default stream) and returns without synchronizing.  Problems visible on
 * the host (bad shapes, NULL or misaligned pointers, a workspace that is too small, an
 * unsupported combination) return an error code before anything is launched.  Problems
 * that only the device can see (a seqlens_k outside [0, cap - curr], a RoPE position
 * beyond rope_len, a pipeline wait that timed out) set bits in *dev_status (if non-NULL;
 * bits are OR-ed in, the caller clears it) and that sequence's outputs are zeros with
 * nothing of it appended.  Kernels never trap or assert.  Calls are reentrant; calls that
 * share a workspace must not overlap on the device.
 */
#ifndef GQA_H_
#define GQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_ABI_VERSION 8

typedef int32_t gqa_status;
#define GQA_OK 0
#define GQA_ERR_INVALID_ARG 1  /* bad shape, attribute, NULL or misaligned pointer */
#define GQA_ERR_UNSUPPORTED 2  /* valid per the op, not implemented by these kernels */
#define GQA_ERR_CAPACITY 3     /* cap_present < curr, cap_past > cap_present, ... */
#define GQA_ERR_CUDA 4         /* a CUDA runtime/driver call failed (launch, tensor map) */
#define GQA_ERR_WORKSPACE 5    /* workspace NULL or smaller than gqa_workspace_bytes() */

/* bits of *dev_status */
#define GQA_DEV_BAD_SEQLEN 1   /* seqlens_k[b] < 0 or > cap - curr (or > cap_past) */
#define GQA_DEV_BAD_ROPE_POS 2 /* past_b + curr > rope_len with do_rotary */
#define GQA_DEV_TIMEOUT 4      /* a bounded pipeline wait gave up; outputs invalid */
#define GQA_DEV_BAD_PAGE 8     /* a block-table entry the step uses is outside [0, num_pages) */
#define GQA_DEV_BOUNDS 16      /* bounds-checked debug build only: a store that would have left
                                  its buffer was skipped (never set by the product build) */
/* The bounds-checked debug build (the package's build(checked=True), compiled with
 * -DGQA_BOUNDS_CHECK into its own folder) has the same entry points; every global store of
 * its kernels is checked against the extent of its buffer, derived from the call.  It also
 * exports the gqa_test_bounds_check probe: given a device int32 [64] buffer and a status
 * word, it makes one store inside and one past a declared extent of 32 elements, so that a
 * test sees the second store skipped and GQA_DEV_BOUNDS set. */

typedef enum { GQA_F32 = 0, GQA_F16 = 1, GQA_BF16 = 2 } gqa_dtype;

/* Op attributes and shapes ([P1], [P2], [P4]). */
typedef struct gqa_params {
  int32_t batch;        /* B >= 1 */
  int32_t q_heads;      /* Hq >= 1, divisible by kv_heads */
  int32_t kv_heads;     /* Hkv >= 1 */
  int32_t head_dim;     /* D: 64 or 128 */
  int32_t q_len;        /* curr >= 1: prompt length (prefill) or new tokens (decode) */
  int32_t cap_past;     /* rows per (b, kv head) of past_k/past_v (ignored when aliased) */
  int32_t cap_present;  /* rows per (b, kv head) of present_k/present_v */
  int32_t rope_len;     /* rows of cos/sin_cache (do_rotary only) */
  int32_t dtype;        /* gqa_dtype of q, k, v, caches, cos/sin and out */
  float scale;          /* score scale; 0 means 1/sqrt(D); must be >= 0 */
  float softcap;        /* 0 means off; else > 0 */
  int32_t window;       /* local_window_size: -1 = none, else >= 1 */
  int32_t causal;       /* 1 = bottom-right causal band, 0 = none */
  int32_t do_rotary;    /* 1 = rotate q and k with cos/sin_cache */
  int32_t rotary_interleaved; /* must be 0 (half-split pairs only) */
  int32_t smooth_softmax;     /* 1 = zero sink when head_sink is NULL */
  int32_t kv_ring;            /* 1 = present is a ring of cap_present slots (see below) */
  int32_t v_head_dim;         /* Dv: 0 = head_dim, else 64 or 128 ([P4] "Layouts and
                                 semantics"); Dv != D only with the contiguous cache
                                 (kv_ring 0, not the paged entry point), else
                                 GQA_ERR_UNSUPPORTED */
} gqa_params;

/* Bytes of device workspace that gqa_attention_prefill / gqa_attention_decode need for
 * these params (the larger of the two), plus, for params with more than one query token
 * that the tensor-core prefill can take, room for a boolean mask's block map
 * (gqa_attention_prefill_masked).  Depends only on the params.  The workspace must be
 * zero-filled before its first use; every call leaves its counters at zero again.
 * Returns 0 for params that fail validation. */
size_t gqa_workspace_bytes(const gqa_params *p);

/* Prefill / first prompt ([P2] "What changed"; [P4] "Compute paths"): RoPE (optional) and
 * append of the curr new tokens, then attention of all curr query rows over present.
 * bf16/f16 run the tensor-core kernel (tcgen05 + TMEM + TMA), f32 the fp32 SIMT kernel.
 * seqlens_k may hold any valid past length (a prompt continued over a non-empty cache).
 * k == NULL and v == NULL selects attention only: present must already hold the step's
 * rows, q is used as given (already rotated), do_rotary must be 0 and past_k/past_v,
 * cos/sin_cache are ignored. */
gqa_status gqa_attention_prefill(const gqa_params *p, const void *q, const void *k, const void *v,
                                 const void *past_k, const void *past_v, const int32_t *seqlens_k,
                                 const void *cos_cache, const void *sin_cache, const float *head_sink,
                                 void *out, void *present_k, void *present_v, void *workspace,
                                 size_t workspace_bytes, int32_t *dev_status, void *stream);

/* Decode step ([P1] "Sliding window" generate branch, multi-token decode; [P2] decode
 * steps): same arguments and semantics as gqa_attention_prefill, executed by the split-KV
 * kernel: each CTA owns all G*curr query rows of one (b, kv head) and one chunk of its
 * visible keys and reads each K/V byte once.  The partial (max, sum, acc) of a group's
 * chunks are merged in distributed shared memory when the chunks form one thread-block
 * cluster (2..8 chunks, launch of one wave), else by the last CTA of the group through the
 * workspace.  For G*curr > 64 (D=64) or > 32 (D=128 or Dv != D), or f32, the fp32 SIMT
 * kernel runs. */
gqa_status gqa_attention_decode(const gqa_params *p, const void *q, const void *k, const void *v,
                                const void *past_k, const void *past_v, const int32_t *seqlens_k,
                                const void *cos_cache, const void *sin_cache, const float *head_sink,
                                void *out, void *present_k, void *present_v, void *workspace,
                                size_t workspace_bytes, int32_t *dev_status, void *stream);

/* RoPE + append alone ([P2] "What changed"): writes present rows [past_b, total_b) (K
 * rotated when do_rotary), copies rows [0, past_b) when present does not alias past, and
 * writes the rotated queries to q_rot (may be NULL; a plain copy when do_rotary == 0).
 * Results are bit-exact: each product and sum is rounded to fp32, then the result to the
 * dtype with ties to even. */
gqa_status gqa_rope_append_kv(const gqa_params *p, const void *q, const void *k, const void *v,
                              const void *past_k, const void *past_v, const int32_t *seqlens_k,
                              const void *cos_cache, const void *sin_cache, void *q_rot, void *present_k,
                              void *present_v, int32_t *dev_status, void *stream);

/* Decode without a workspace.  No page describes this entry point; it exists for
 * callers that cannot allocate device memory where they run attention -- a plugin hosted by
 * an inference engine that owns all device memory and gives its plugins no allocator, or a
 * latency-critical loop in which a cudaMalloc (which can synchronize the device) is not
 * acceptable.  Same arguments and semantics as gqa_attention_decode, without the workspace:
 * the library keeps the scratch in one static device array of GQA_NOALLOC_SCRATCH_BYTES
 * bytes, which every GPU that loads the library holds until the process exits.  Params
 * that need more (gqa_workspace_bytes(p) > GQA_NOALLOC_SCRATCH_BYTES) return
 * GQA_ERR_WORKSPACE with nothing launched.  The first call on each device looks up the
 * array's device address with that device current; make that first call before any stream
 * capture.  Every call clears the counters it relies on and reuses the same array, which
 * keeps the previous call's contents, so calls that overlap on the GPU (other streams,
 * other threads) race on it and must be serialized by the caller.  Nothing in this call
 * allocates or frees memory. */
#define GQA_NOALLOC_SCRATCH_BYTES (32u << 20)
gqa_status gqa_attention_decode_noalloc(const gqa_params *p, const void *q, const void *k, const void *v,
                                        const void *past_k, const void *past_v, const int32_t *seqlens_k,
                                        const void *cos_cache, const void *sin_cache, const float *head_sink,
                                        void *out, void *present_k, void *present_v, int32_t *dev_status,
                                        void *stream);

/* Decode over a paged KV cache ([P3] Summary: a cell cache whose slots belong to sequences
 * and are masked, not evicted).  The cache is a pool of pages of 64 positions,
 * k_pool/v_pool [num_pages, Hkv, 64, D] (dtype), shared by all sequences; block_table is
 * int32 [B, max_pages] on the device, entry n of row b naming the page that holds positions
 * [64n, 64n + 64) of sequence b.  p->cap_present must be 64 * max_pages (the logical
 * capacity of a sequence); p->cap_past is ignored and p->kv_ring must be 0.  The step's rows
 * are written into their pages (in place: there is no separate past).  Only the entries for
 * the positions the step reads or writes ([first page of the band, last new position]) are
 * read; a sequence for which one of them lies outside [0, num_pages) gets zeros, nothing
 * written, and GQA_DEV_BAD_PAGE.  Otherwise the same semantics, kernel, workspace
 * (gqa_workspace_bytes) and errors as gqa_attention_decode, including k = v = NULL for
 * attention only; shapes outside the split-KV kernel's envelope return GQA_ERR_UNSUPPORTED. */
gqa_status gqa_attention_decode_paged(const gqa_params *p, const void *q, const void *k, const void *v,
                                      const int32_t *seqlens_k, const int32_t *block_table, int32_t max_pages,
                                      int32_t num_pages, const void *cos_cache, const void *sin_cache,
                                      const float *head_sink, void *out, void *k_pool, void *v_pool,
                                      void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                      void *stream);

/* Prefill (a prompt, or a chunk of one over the pages already filled) into the same paged
 * cache: the arguments, pages, table rules and errors of gqa_attention_decode_paged, with
 * gqa_attention_prefill's semantics and kernels: the RoPE/append kernel writes the step's
 * rows through the table (every page of the step's band checked first, the same decision
 * as the attention kernel's), then the tensor-core prefill reads the band as 128-position
 * tiles, each two pages.  bf16/f16 only (f32 returns GQA_ERR_UNSUPPORTED).  The workspace
 * holds the rotated queries when do_rotary (gqa_workspace_bytes). */
gqa_status gqa_attention_prefill_paged(const gqa_params *p, const void *q, const void *k, const void *v,
                                       const int32_t *seqlens_k, const int32_t *block_table, int32_t max_pages,
                                       int32_t num_pages, const void *cos_cache, const void *sin_cache,
                                       const float *head_sink, void *out, void *k_pool, void *v_pool,
                                       void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                       void *stream);

/* Attention mask ([P4] "Layouts and semantics": boolean and FLOAT additive broadcast
 * masks next to the bottom-right causal band; [P2] "What changed": attention_bias summed
 * with the band).  Element [b][hq][i][j] (batch, q head, new token, key = absolute
 * position) is at data + b*stride_b + hq*stride_h + i*stride_i + j elements; a stride of 0
 * broadcasts that dimension, and the keys are contiguous.  kind GQA_MASK_KEEP: uint8, zero
 * removes the key from the row's softmax exactly like the band does.  kind GQA_MASK_ADD:
 * values of the params' dtype added to the scaled score before the softcap (score, mask,
 * softcap, softmax).  keys: the extent of the key dimension; a sequence with
 * seqlens_k + q_len > keys is rejected (GQA_DEV_BAD_SEQLEN, zeros).  The band, the sink and
 * the fully-masked-row rule are unchanged. */
#define GQA_MASK_KEEP 1
#define GQA_MASK_ADD 2
typedef struct gqa_mask {
  const void *data;
  int32_t kind;
  int32_t keys;
  int64_t stride_b, stride_h, stride_i;
} gqa_mask;

/* Decode step with an attention mask: gqa_attention_decode's arguments and semantics plus
 * *mask (device data, host struct).  Shapes inside the split-KV kernel's envelope run it
 * (ring caches, kv_ring, are allowed there; the mask stays indexed by absolute position);
 * f32 params and other shapes run the CUDA-core kernel (a ring then returns
 * GQA_ERR_UNSUPPORTED).  An additive mask's data is aligned to its element size. */
gqa_status gqa_attention_decode_masked(const gqa_params *p, const gqa_mask *mask, const void *q, const void *k,
                                       const void *v, const void *past_k, const void *past_v,
                                       const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                       const float *head_sink, void *out, void *present_k, void *present_v,
                                       void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                       void *stream);

/* Prefill (or any step) with an attention mask: gqa_attention_prefill's arguments and
 * semantics plus *mask, as for gqa_attention_decode_masked.  bf16/f16 with head_dim 64 or
 * 128 and a mask whose data address and non-zero strides (in bytes) are multiples of 16
 * run the tensor-core kernel, which stages the mask by TMA; any other mask, and f32, run
 * the CUDA-core kernel (same results within the dtype's tolerance, slower).  A boolean
 * (GQA_MASK_KEEP) mask on the tensor-core kernel skips the 128-key tiles in which it keeps
 * no key of a 128-row query tile ([P4] "Compute paths": an all-false block is skipped) when
 * workspace_bytes >= gqa_workspace_bytes(p): a first kernel writes the mask's block map into
 * the workspace.  With a smaller workspace every tile is streamed; the results are the same
 * (keys the mask removes never contribute; a skipped tile is never read at all). */
gqa_status gqa_attention_prefill_masked(const gqa_params *p, const gqa_mask *mask, const void *q, const void *k,
                                        const void *v, const void *past_k, const void *past_v,
                                        const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                        const float *head_sink, void *out, void *present_k, void *present_v,
                                        void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                        void *stream);

/* Attention over a K/V cache with padding ([P4] "Layouts and semantics": the opset-24
 * nonpad_kv_seqlen input; "Compute paths": padding frontiers skip unavailable blocks).
 * nonpad_kv_seqlen is int64 [B] on the device (8-byte aligned): sequence b has n_b valid
 * keys, rows [0, n_b) of k_cache [B, Hkv, cap_present, D] / v_cache [B, Hkv, cap_present,
 * Dv]; rows at or past n_b are padding and are never read.  The q_len queries
 * ([B, q_len, Hq*D], used as given: do_rotary must be 0) are the last q_len of the n_b valid
 * tokens, so query i sits at absolute position n_b - q_len + i and the causal band, the
 * window, the sink, the softcap and the fully-masked-row rule apply as for
 * gqa_attention_prefill with seqlens_k = n_b - q_len (attention only: nothing is
 * appended).  A sequence with n_b < q_len or n_b > cap_present gets zeros and
 * GQA_DEV_BAD_SEQLEN.  kv_ring must be 0.  Kernel: the split-KV decode kernel when its
 * envelope holds the shape, else the tensor-core prefill (bf16/f16) or the fp32 kernel; the
 * workspace is gqa_workspace_bytes(p).  Errors as for gqa_attention_prefill. */
gqa_status gqa_attention_nonpad(const gqa_params *p, const int64_t *nonpad_kv_seqlen, const void *q,
                                const void *k_cache, const void *v_cache, const float *head_sink, void *out,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/* f8 KV cache.  The pages leave a quantized cache out of their own designs ([P1] puts
 * i8/i4/f8 KV out of its scope; [P2] "What changed" rejects quantized KV); this is the
 * plainest reading for an f8 cache.  present_k [B, Hkv, cap_present, D] and present_v
 * [B, Hkv, cap_present, Dv] hold one byte per element: an E4M3 code (1 sign, 4 exponent
 * bits with bias 7, 3 fraction bits, no infinities, S.1111.111 = NaN, largest magnitude
 * 448).  The stored value of an element is code * scale, with k_scale[h] / v_scale[h]
 * (fp32, device, [Hkv]) the scales of kv head h.  The step's K (rotated and rounded to the
 * dtype first, as without quantization) and V rows are appended as the codes of
 * fp32(x) / scale: nearest, ties to even, saturating at +-448 (infinity too), NaN to NaN.
 * Attention is the op's definition over the stored values.  The cache is updated in place
 * (no separate past; k = v = NULL for attention only); q, out, k, v, cos/sin keep the
 * params' dtype; kv_ring returns GQA_ERR_UNSUPPORTED.  Same workspace (gqa_workspace_bytes),
 * status and errors as gqa_attention_decode / gqa_attention_prefill.  Decode with D = Dv =
 * 128 inside the split-KV kernel's envelope runs that kernel (f8 tiles by TMA, converted to
 * f16 MMA operands); every other shape runs the CUDA-core kernel. */
gqa_status gqa_attention_decode_q8(const gqa_params *p, const void *q, const void *k, const void *v,
                                   const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                   const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                   uint8_t *present_k, uint8_t *present_v, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream);
gqa_status gqa_attention_prefill_q8(const gqa_params *p, const void *q, const void *k, const void *v,
                                    const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                    const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                    uint8_t *present_k, uint8_t *present_v, void *workspace, size_t workspace_bytes,
                                    int32_t *dev_status, void *stream);

/* int8 KV cache: the same layouts, scales, arguments, kernels and errors as the f8 calls
 * above, with each element a two's-complement code in [-128, 127] whose stored value is
 * code * scale.  The pages define no integer format either; this is the plainest reading,
 * the ONNX QuantizeLinear convention with a zero point of 0: the step's rows are appended
 * as round(fp32(x) / scale), ties to even, saturating at -128 and 127 (infinities too), and
 * NaN, which that convention leaves undefined, as 0.  The split-KV kernel converts the codes
 * to f16 exactly (every int8 value is an f16 value). */
gqa_status gqa_attention_decode_i8(const gqa_params *p, const void *q, const void *k, const void *v,
                                   const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                   const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                   int8_t *present_k, int8_t *present_v, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream);
gqa_status gqa_attention_prefill_i8(const gqa_params *p, const void *q, const void *k, const void *v,
                                    const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                                    const float *head_sink, const float *k_scale, const float *v_scale, void *out,
                                    int8_t *present_k, int8_t *present_v, void *workspace, size_t workspace_bytes,
                                    int32_t *dev_status, void *stream);

/* Static description of a status code. */
const char *gqa_status_string(gqa_status s);

/* GQA_ABI_VERSION of the loaded library. */
int32_t gqa_abi_version(void);

/* Test hook for the failure path ([P4] "Scheduling, precision, and invariants": invalid
 * situations fail explicitly).  Every pipeline wait in the tensor-core prefill and split-KV
 * decode kernels is bounded (about 2 s by default); a wait that gives up sets
 * GQA_DEV_TIMEOUT, lets the copies and MMAs its CTA already issued land (those waits keep the
 * full bound), frees the CTA's tensor memory and returns, and the call's outputs are then
 * invalid.  With cycles > 0, every later launch of those kernels (in this process) first
 * waits on an mbarrier that nothing completes and bounds its pipeline waits by `cycles` SM
 * cycles, so that this path runs deterministically; the workspace stays usable for the next
 * call.  cycles == 0 restores normal operation; cycles < 0 returns GQA_ERR_INVALID_ARG.
 * Not for production use. */
gqa_status gqa_test_stall_waits(int64_t cycles);

#ifdef __cplusplus
}
#endif
#endif /* GQA_H_ */

/*
 * attn.h — C ABI of the GB300 (sm_103a) fused softmax-attention library.
 *
 * The operation is softmax attention O = softmax(Q K^T * scale + mask) V,
 * computed with online softmax so that the score matrix S is never stored,
 * plus the per-row log-sum-exp LSE = ln sum_j exp(s_ij).
 *
 * Sources (web pages on softmax attention):
 *   [DEVLOG] "Agent 帮我写 CUDA：一个 Softmax Attention 算子的开发全记录", a fp32
 *            softmax-attention CUDA development log: section 二 "参考基线" (the
 *            operator on [B,H,N,D] tensors and its SDPA reference), section 三
 *            "Step 1：Naive 版本" (raw-pointer kernel signature, a shared library
 *            called from Python), section 四 "Tiled Attention 的核心思想" (the
 *            online-softmax recurrence and the tile loop).
 *   [ASK]    "Ask, Don't Equip: Question-Driven Coding Agents for Deep Kernel
 *            Optimization", section "研究动机": GQA, causal / sliding-window masks
 *            and split-KV decode as parts of the attention forward's feature
 *            surface.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or copies device memory and never synchronises,
 *     except in attn_get_device_error().  Work is queued on `stream`
 *     (NULL = the legacy default stream) and runs asynchronously.
 *   - Tensors are dense and contiguous, row-major in the order their shape is
 *     written.  Every tensor pointer must be 16-byte aligned.
 *   - Masking: key j is visible to query i iff j < Nk, and, when causal != 0,
 *     j <= i + Nk - Nq (bottom-right aligned: j <= i when Nq == Nk), and, when
 *     window > 0, j > i + Nk - Nq - window (the last `window` keys up to the
 *     diagonal).  window <= 0 disables the window.  There is no additive mask
 *     tensor.  A query row that sees no key gets O = 0 and LSE = -inf.
 *   - GQA: query head h reads KV head h / (Hq / Hkv); Hq must be a multiple of
 *     Hkv (Hkv == Hq is plain multi-head attention, Hkv == 1 multi-query).
 *   - LSE is the natural logarithm of the softmax denominator of the scaled,
 *     masked scores, in fp32.
 *   - Return value: ATTN_OK (0) or a negative ATTN_ERR_* code.  Argument errors
 *     are detected on the host before anything is queued.  Errors found on the
 *     device (an expired bounded wait, an out-of-range sequence length) are
 *     recorded in a per-device error word and reported by the next call to
 *     attn_get_device_error().
 */
#ifndef SOFTMAX_ATTENTION_ATTN_GB300_ATTN_H
#define SOFTMAX_ATTENTION_ATTN_GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t;

enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_NULL = -1,        /* a required pointer is NULL                              */
  ATTN_ERR_DIM = -2,         /* a size is non-positive or too large                     */
  ATTN_ERR_GQA = -3,         /* Hq is not a multiple of Hkv                             */
  ATTN_ERR_HEAD_DIM = -4,    /* head dimension D not supported by this entry point      */
  ATTN_ERR_ALIGN = -5,       /* a tensor pointer is not 16-byte aligned                 */
  ATTN_ERR_SCALE = -6,       /* scale is not finite or not > 0                          */
  ATTN_ERR_CUDA = -7,        /* a CUDA runtime / launch error                           */
  ATTN_ERR_TIMEOUT = -8,     /* a bounded device-side wait expired (kernel gave up)     */
  ATTN_ERR_DEVICE = -9,      /* the current device is not an sm_103 GPU                */
  ATTN_ERR_SEQLEN = -10,     /* a decode sequence length is < 1 or > Nk_max (device)   */
  ATTN_ERR_CHUNK = -11,      /* split-KV chunk size not supported                       */
  ATTN_ERR_CAPACITY = -12,   /* a size exceeds a fixed capacity of the entry point      */
  ATTN_ERR_PAGE = -13        /* a block-table entry in use is outside [0, num_pages)    */
};

/*
 * attn_fwd — bf16 fused attention forward on tensor cores (tcgen05 / TMEM).
 *   [DEVLOG] 二 "参考基线" (operator), 四 "Tiled Attention 的核心思想" (online
 *   softmax over K/V tiles); [ASK] "研究动机" (GQA, causal, sliding window).
 *
 *   q   : bf16 [B, Hq,  Nq, D]        k, v : bf16 [B, Hkv, Nk, D]
 *   o   : bf16 [B, Hq,  Nq, D] (out)  lse  : fp32 [B, Hq, Nq] (out; may be NULL)
 *   D must be 64 or 128.  Scores and accumulation are fp32; P is rounded to bf16
 *   before the P V product; O is rounded to bf16 (round-to-nearest-even).
 *   scale multiplies Q K^T (1/sqrt(D) for standard attention).
 *   Errors: ATTN_ERR_NULL, _DIM, _GQA, _HEAD_DIM, _ALIGN, _SCALE, _DEVICE, _CUDA.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int Nq, int Nk, int D,
             float scale, int causal, int window, attn_stream_t stream);

/*
 * attn_fwd_softcap_sink — attn_fwd with a softcap on the scores and one sink
 * logit per query head.   [ASK] "研究动机" (softcap and attention-sink masks on
 * the feature list; the pages give no formulas).
 *
 *   softcap : c > 0 maps each scaled score s = scale * q.k to c * tanh(s / c)
 *             before the softmax (masked scores stay masked); c <= 0 disables
 *   sinks   : device float32 [Hq] or NULL.  sinks[h] (natural-log units, may be
 *             -inf) joins the softmax denominator of every row of query head h
 *             without a value: P_ij = exp(s_ij) / (sum_j exp(s_ij) + exp(sinks[h]))
 *             and LSE_i = ln(sum_j exp(s_ij) + exp(sinks[h])); a row with no
 *             visible key gets O = 0 and LSE = sinks[h]
 *   Every other argument, layout and result is that of attn_fwd (bf16; D 64 or
 *   128; causal, window).
 *   Errors: as attn_fwd, plus ATTN_ERR_SCALE for a softcap that is not finite
 *   and ATTN_ERR_ALIGN for a sinks pointer that is not 4-byte aligned.
 */
int attn_fwd_softcap_sink(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                          int window, float softcap, const float* sinks, attn_stream_t stream);

/*
 * attn_fwd_fp16 — fp16 variant of attn_fwd (same kernel, fp16 tensor-core
 * operands).  [ASK] "研究动机" (bf16 / fp16 / fp8 precisions on the feature
 * surface).  Same shapes, masks, D and error codes as attn_fwd with fp16 q, k,
 * v and o; P is rounded to fp16 before the P V product; O is rounded to fp16.
 */
int attn_fwd_fp16(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int Hq, int Hkv, int Nq, int Nk, int D,
                  float scale, int causal, int window, attn_stream_t stream);

/*
 * attn_fwd_fp8_workspace_size — bytes of device workspace attn_fwd_fp8 needs:
 * a bf16 copy of V, B * Hkv * Nk * D * 2.  Returns 0 for invalid sizes.
 */
size_t attn_fwd_fp8_workspace_size(int B, int Hkv, int Nk, int D);

/*
 * attn_fwd_fp8 — fused attention forward on fp8 (E4M3) Q, K and V.
 *   [ASK] "局限与改进" (fp8 dense prefill among the weakest scenarios) and
 *   "未来方向" (fp8 among the work still open); the operator is that of attn_fwd.
 *
 *   q    : uint8 [B, Hq,  Nq, D]  k, v : uint8 [B, Hkv, Nk, D], one OCP FP8
 *          E4M3 code per element (sign bit 7, exponent bits 6-3 with bias 7,
 *          mantissa bits 2-0; S.1111.111 is NaN).  An element's value is its
 *          E4M3 value times q_scale, k_scale or v_scale (per-tensor, host floats).
 *   o    : bf16 [B, Hq, Nq, D] (out)   lse : fp32 [B, Hq, Nq] (out; may be NULL)
 *   workspace : device, attn_fwd_fp8_workspace_size(B, Hkv, Nk, D) bytes, owned
 *          by the caller; overwritten (it receives V widened to bf16).
 *   D must be 128.  S = Q K^T runs on the E4M3 codes (tensor cores, fp32
 *   accumulation) and is scaled by scale * q_scale * k_scale; P is rounded to
 *   bf16 and multiplied by the exact bf16 copy of V; O is multiplied by v_scale
 *   and rounded to bf16.  Masks, GQA and LSE are those of attn_fwd.
 *   Errors: as attn_fwd; ATTN_ERR_NULL / _ALIGN also for the workspace;
 *   ATTN_ERR_SCALE also for a q_scale, k_scale or v_scale that is not finite or
 *   not > 0, or a product scale * q_scale * k_scale that is not a finite
 *   positive float.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                 float v_scale, void* o, float* lse, void* workspace,
                 int B, int Hq, int Hkv, int Nq, int Nk, int D,
                 float scale, int causal, int window, attn_stream_t stream);

/*
 * attn_fwd_varlen — bf16 forward on a ragged batch (packed, token-major).
 *   [ASK] "研究动机" (ragged batches on the feature surface).
 *
 *   q, o : bf16 [total_q, Hq, D]      k, v : bf16 [total_k, Hkv, D]
 *   lse  : fp32 [Hq, total_q] (may be NULL)
 *   cu_seqlens_q, cu_seqlens_k : int32 [B + 1] (device), non-decreasing, starting
 *   at 0: sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and
 *   key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1.  Masks and GQA act within a
 *   sequence (causal is bottom-right aligned per sequence).  max_seqlen_q must
 *   be >= every query length; an empty sequence is allowed.  A slice outside
 *   [0, total) or longer than max_seqlen_q is skipped and reported as
 *   ATTN_ERR_SEQLEN in the device error word.  D must be 64 or 128.
 *   Errors: as attn_fwd.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens_q, const int* cu_seqlens_k,
                    int B, int Hq, int Hkv, int max_seqlen_q, int total_q, int total_k, int D,
                    float scale, int causal, int window, attn_stream_t stream);

/*
 * attn_fwd_fp32 — fp32 fused attention forward on the FP32 SIMT pipes.
 *   [DEVLOG] 三 (fp32 [B,H,N,D] operator), 四 (tiled online softmax),
 *   五 (16-byte vector loads, padded shared-memory rows).
 *
 *   Same shapes, masks and error codes as attn_fwd, with fp32 q, k, v, o.
 *   D must be 32, 64 or 128.  No reduced-precision arithmetic is used.
 */
int attn_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse,
                  int B, int Hq, int Hkv, int Nq, int Nk, int D,
                  float scale, int causal, int window, attn_stream_t stream);

/*
 * attn_decode_workspace_size — bytes of device workspace that
 * attn_decode_splitkv fills and attn_decode_combine reads:
 *   fp32 O_part [B, Hq, S_max, D] followed by fp32 LSE_part [B, Hq, S_max],
 *   S_max = ceil(Nk_max / chunk).  Returns 0 for invalid sizes.
 */
size_t attn_decode_workspace_size(int B, int Hq, int D, int Nk_max, int chunk);

/*
 * attn_decode_splitkv — split-KV decode, partial step.   [ASK] "研究动机"
 *   (split-KV decode); each chunk's result is the tiled online softmax of
 *   [DEVLOG] 四 restricted to the chunk's keys.
 *
 *   q        : bf16 [B, Hq, D]              (one query token per sequence)
 *   k_cache  : bf16 [B, Nk_max, Hkv, D]     v_cache : bf16 [B, Nk_max, Hkv, D]
 *   seqlens  : int32 [B] (device)           sequence b uses rows 0..seqlens[b]-1
 *   workspace: device buffer of attn_decode_workspace_size(B, Hq, D, Nk_max, chunk)
 *              bytes.  For each b, head h and chunk c < ceil(seqlens[b]/chunk)
 *              (keys c*chunk .. min((c+1)*chunk, seqlens[b]) - 1) it receives the
 *              chunk's normalised output O_c and its LSE_c; other entries are
 *              left untouched.
 *   D must be 64 or 128; Hq / Hkv must be 1, 2, 4, 8, 16 or 32 (32 with Hkv = 1
 *   is multi-query decode); chunk must be a multiple of 64 in [64, 1024].  The
 *   chunk's scores for all query heads of a KV head are held in shared memory,
 *   so a combination whose shared memory would exceed the per-block limit
 *   returns ATTN_ERR_CAPACITY (D = 128, Hq / Hkv = 32 fits every chunk size).  A seqlens[b] outside [1, Nk_max] sets ATTN_ERR_SEQLEN in
 *   the device error word and that sequence is skipped.
 *   Errors: ATTN_ERR_NULL, _DIM, _GQA, _HEAD_DIM, _ALIGN, _SCALE, _CHUNK,
 *   _DEVICE, _CUDA.
 */
int attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                        const int* seqlens, void* workspace,
                        int B, int Hq, int Hkv, int Nk_max, int D,
                        float scale, int chunk, attn_stream_t stream);

/*
 * attn_decode_splitkv_paged — split-KV decode, partial step, on a paged KV
 * cache.   [ASK] "研究动机" (paged and contiguous KV caches, split-KV decode).
 *
 *   k_pages, v_pages : bf16 [num_pages, page_size, Hkv, D]   (a shared page pool)
 *   block_table      : int32 [B, max_pages] (device); key j of sequence b is row
 *                      j % page_size of page block_table[b, j / page_size]
 *   Other arguments, the workspace layout and the results are those of
 *   attn_decode_splitkv with Nk_max = max_pages * page_size (size the
 *   workspace and call attn_decode_combine with that Nk_max).  page_size must
 *   be a multiple of 64 (a 64-key tile never straddles two pages).  Only the
 *   block-table entries of pages that hold keys j < seqlens[b] are read; an
 *   entry outside [0, num_pages) sets ATTN_ERR_PAGE in the device error word
 *   (that tile reads zeros).
 *   Errors: as attn_decode_splitkv, plus ATTN_ERR_DIM for a page_size that is
 *   not a positive multiple of 64.
 */
int attn_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int* block_table, const int* seqlens, void* workspace,
                              int B, int Hq, int Hkv, int num_pages, int page_size, int max_pages,
                              int D, float scale, int chunk, attn_stream_t stream);

/*
 * attn_bwd_workspace_size — bytes of device workspace attn_bwd needs:
 *   2 * B * Hq * ceil(Nq / 128) * 128 * 4 (per query, padded to 128 rows per
 *   head: -LSE * log2(e) and -scale * D with D = rowsum(dO * O)).
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Nq);

/*
 * attn_bwd — attention backward: the gradients of attn_fwd's O with respect to
 * Q, K and V for an upstream gradient dO.   [DEVLOG] 二 (the forward
 * O = softmax(scale Q K^T) V); [ASK] "研究动机" (forward only there; the
 * backward pass is named as the next piece of work).
 *
 *   q, o, dout : bf16 [B, Hq, Nq, D]; k, v : bf16 [B, Hkv, Nk, D]
 *   lse        : float32 [B, Hq, Nq], the forward's LSE (natural log; -inf for
 *                rows with no visible key) for the same q, k, v, scale, causal
 *   dq         : float32 [B, Hq, Nq, D] (output; zeroed, then accumulated)
 *   dk, dv     : bf16 [B, Hkv, Nk, D] (outputs; K/V gradients of a KV head sum
 *                over the query heads that read it)
 *   workspace  : device buffer of attn_bwd_workspace_size(B, Hq, Nq) bytes
 *   causal, window : the forward's masks, as in attn_fwd (bottom-right causal;
 *                window > 0 keeps the last `window` keys up to the diagonal)
 *   D must be 64 or 128.  All device pointers 16-byte aligned, contiguous; the
 *   caller owns every buffer.  Asynchronous on `stream`.
 *   Errors: ATTN_ERR_NULL, ATTN_ERR_DIM, ATTN_ERR_GQA, ATTN_ERR_HEAD_DIM,
 *   ATTN_ERR_ALIGN, ATTN_ERR_SCALE, ATTN_ERR_CUDA; a bounded wait that runs
 *   out sets ATTN_ERR_TIMEOUT in the device error word.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, float* dq, void* dk, void* dv, void* workspace, int B, int Hq,
             int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
             attn_stream_t stream);

/*
 * attn_decode_splitkv_fp8 — split-KV decode, partial step, on an fp8 KV cache.
 *   [ASK] "研究动机" (bf16/fp16/fp8 data types, fp8-KV decode shapes).
 *
 *   k_cache, v_cache : uint8 [B, Nk_max, Hkv, D] (device), one OCP FP8 E4M3 code
 *                      per element (sign bit 7, exponent bits 6-3 with bias 7,
 *                      mantissa bits 2-0; S.1111.111 is NaN).  The element's
 *                      value is its E4M3 value times k_scale (K) or v_scale (V).
 *   k_scale, v_scale : per-tensor dequantisation scales (host floats, finite, > 0)
 *   q, seqlens, workspace and every other argument, the workspace layout and the
 *   results are those of attn_decode_splitkv (q stays bf16; combine with
 *   attn_decode_combine).  The arithmetic runs in fp32 on the exact decoded
 *   values.  Cache rows at or past seqlens[b] are never weighted, whatever
 *   codes they hold.
 *   Errors: as attn_decode_splitkv; ATTN_ERR_SCALE also for a k_scale or v_scale
 *   that is not finite or not > 0.
 */
int attn_decode_splitkv_fp8(const void* q, const void* k_cache, const void* v_cache,
                            float k_scale, float v_scale, const int* seqlens, void* workspace,
                            int B, int Hq, int Hkv, int Nk_max, int D, float scale, int chunk,
                            attn_stream_t stream);

/*
 * attn_decode_splitkv_paged_fp8 — split-KV decode, partial step, on a paged fp8
 * KV cache.   [ASK] "研究动机" (paged caches, fp8 data types).
 *
 *   k_pages, v_pages : uint8 [num_pages, page_size, Hkv, D] E4M3 codes, values
 *                      as in attn_decode_splitkv_fp8
 *   Every other argument, the block-table rules and the errors are those of
 *   attn_decode_splitkv_paged plus the scale checks of attn_decode_splitkv_fp8.
 */
int attn_decode_splitkv_paged_fp8(const void* q, const void* k_pages, const void* v_pages,
                                  float k_scale, float v_scale, const int* block_table,
                                  const int* seqlens, void* workspace, int B, int Hq, int Hkv,
                                  int num_pages, int page_size, int max_pages, int D, float scale,
                                  int chunk, attn_stream_t stream);

/*
 * attn_decode_combine — split-KV decode, combine step.   [ASK] "研究动机"
 * (split-KV decode: the chunks' partial results are merged into one output).
 * LSE-weighted merge of the chunk results written by attn_decode_splitkv:
 *   M = max_c LSE_c,  w_c = exp(LSE_c - M),  O = sum_c w_c O_c / sum_c w_c,
 *   LSE = M + ln sum_c w_c,   over c < ceil(seqlens[b] / chunk).
 *   o : bf16 [B, Hq, D] (out)        lse : fp32 [B, Hq] (out; may be NULL)
 *   Arguments B, Hq, Nk_max, D, chunk must equal those of the splitkv call.
 *   Errors: as attn_decode_splitkv.
 */
int attn_decode_combine(const void* workspace, const int* seqlens, void* o, float* lse,
                        int B, int Hq, int Nk_max, int D, int chunk,
                        attn_stream_t stream);

/*
 * attn_decode_noalloc — split-KV decode (partial step, then combine step) that
 * allocates nothing and needs no workspace from the caller.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory themselves, e.g. a plugin inside a host runtime that owns the whole
 * device memory pool, or a latency-critical caller that must never reach
 * cudaMalloc.
 *
 *   Arguments, layouts, results and error codes are those of
 *   attn_decode_splitkv followed by attn_decode_combine, with o / lse as the
 *   outputs.  The per-chunk partials live in a scratch array inside the
 *   library image of ATTN_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB); every GPU that
 *   loads this part of the library keeps it until the process exits.  Sizes
 *   needing more scratch than that, i.e.
 *   attn_decode_workspace_size(B, Hq, D, Nk_max, chunk) > 16 MiB, are rejected
 *   with ATTN_ERR_CAPACITY before anything is queued.  Checks run in this
 *   order: NULL pointers (ATTN_ERR_NULL), sizes for which no workspace size
 *   exists (ATTN_ERR_DIM), the capacity (ATTN_ERR_CAPACITY), then the checks
 *   of attn_decode_splitkv and attn_decode_combine.
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress, once per device) and keeps it for the rest of the
 *   process: make that first call before any stream capture, and do not call
 *   this entry point again on a device after cudaDeviceReset() or any other
 *   teardown of its primary context (the kept address then no longer names
 *   the scratch array; the library's device error word is cached the same way).  All calls share the one array, so calls whose kernels
 *   overlap on the GPU (different streams without ordering) race and corrupt
 *   each other's results; calls on one stream are ordered and safe.  Nothing in
 *   the scratch needs to start at zero: every entry the combine step reads is
 *   written by the partial step of the same call.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)
int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                        const int* seqlens, void* o, float* lse,
                        int B, int Hq, int Hkv, int Nk_max, int D,
                        float scale, int chunk, attn_stream_t stream);

/*
 * attn_get_device_error — synchronises `stream`, then returns and clears the
 * current device's error word (ATTN_OK if no kernel reported an error).  A
 * CUDA error seen while synchronising is returned as ATTN_ERR_CUDA.
 */
int attn_get_device_error(attn_stream_t stream);

/* attn_strerror — static, human-readable text for a status code. */
const char* attn_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* SOFTMAX_ATTENTION_ATTN_GB300_ATTN_H */

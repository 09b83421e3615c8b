// attn_bwd.cu — bf16 attention backward (dQ, dK, dV) for sm_103a on tcgen05.
//
// The gradients of the forward of "Agent 帮我写 CUDA：一个 Softmax Attention
// 算子的开发全记录" (section 二: O = softmax(scale Q K^T) V) for an upstream
// gradient dO, the backward pass named as missing work in "Ask, Don't Equip:
// ..." (section "研究动机", forward only; "then the backward pass"):
//
//   P = exp(scale Q K^T - LSE)   (LSE from the forward; masked entries 0)
//   dV = P^T dO      dP = dO V^T      D = rowsum(dO * O) = rowsum(P * dP)
//   dS = P * (dP - D)      dQ = scale dS K      dK = scale dS^T Q
//   (K and V gradients of a KV head sum over the query heads that read it).
//
// Design: one CTA per (batch, KV head, 128-key tile j); it keeps K_j and V_j
// in shared memory and dK_j, dV_j in tensor memory while it walks every query
// head of the KV head's group and every 128-query tile i that sees the key
// tile.  With the keys on the tensor-memory lanes:
//   * S^T = K_j Q_i^T and dP^T = V_j dO_i^T (M = 128 keys, N = 128 queries);
//   * eight row warps, two per lane quarter (thread r owns key r; the two
//     warps of a quarter take queries [0,64) and [64,128)), form P^T as soon
//     as S^T is done (while the dP^T MMAs run) and dS^T = scale P^T (dP^T - D)
//     as soon as dP^T is done (while the dV MMAs run), in fp32; P^T goes as
//     bf16 pairs into the first half of the S^T columns each warp read, dS^T
//     as bf16 into shared memory;
//   * dV_j += P^T dO_i (A from tensor memory, the TS form) and dK_j += dS^T Q_i
//     (A from shared memory);
//   * dQ_i = dS K_j (M = 128 queries, N = 128 head dims; both operands
//     MN-major in shared memory: dS^T and K_j as they lie) over the dP^T
//     columns, which the row warps have read before handing dS^T over; four
//     more warps read it (thread r owns query
//     r), free the columns for the next dP^T, stage it as fp32 in the Q/dO
//     stage the step has finished with (128-byte swizzled 32 x 32 boxes) and
//     add it to the fp32 dQ with TMA reduce-add copies while the next step
//     runs.  (Per-thread global atomics here would fill the load/store queue
//     that the row warps' shared-memory loads share.)  The stage is handed
//     back to the TMA warp once the copies have read it;
//   * one TMA warp streams Q_i, dO_i (and the per-query -LSE*log2(e) and
//     -scale*D vectors, prepared by attn_bwd_prep_kernel) through a 2-stage ring; one
//     thread issues every MMA.  128-query steps keep every MMA at N = 128 or
//     K = 128: a 128 x 64 x 16 MMA takes almost as long to issue and run as a
//     128 x 128 x 16 one.
// Tensor memory (512 columns): S^T / P^T [0,128), dP^T / dQ [128,256),
// dV [256,384), dK [384,512).  Shared memory: the 1024-byte aligned operand
// block (K_j, V_j, two Q/dO stages, dS^T) fills all but 3 KB of the 227 KB, so
// the barriers sit in front of it when the alignment padding has room and
// behind it otherwise, next to the per-stage vectors.  Every wait is bounded
// (see ptx.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace bwd {

constexpr int BK = 128;                          // keys per CTA
constexpr int BQ = 128;                          // queries per step
constexpr int NS = 2;                            // Q / dO ring stages
constexpr int KSLAB = BK * 128;                  // 64-column slab of a 128-row tile (16 KB)
constexpr int QSLAB = BQ * 128;                  // 64-column slab of a 128-row tile (16 KB)
constexpr int VEC_BYTES = 2 * BQ * 4;            // -LSE*log2(e)[128], -scale*D[128]
constexpr int NUM_BARS = 1 + 2 * NS + 8;
constexpr int SMALL_BYTES = 128;                 // barriers + misc words
static_assert(NUM_BARS * 8 + 16 <= SMALL_BYTES, "small block");
constexpr int SMEM_ALLOC = 227 * 1024;
constexpr int NROW = 8;                          // row warps 0..7: lane quad = warp % 4, query half = warp / 4
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int WARP_DQ0 = 10;                     // warps 10..13 read dQ out (lane quad = warp % 4)
constexpr int NTHREADS = 14 * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 384, COL_DQ = COL_DP;

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D; bit 15 / 16 set
// the A / B operand MN-major.
constexpr uint32_t idesc(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}
constexpr uint32_t ID_ST = idesc(BK, BQ, 0, 0);   // S^T, dP^T: K / V and Q / dO, both K-major
static_assert(BQ == 128 && BK == 128, "tile shapes");

// Shared-memory layout and head-dimension-dependent MMA shapes for head dimension HD
// (64 or 128): K_j, V_j and each stage's Q_i, dO_i are HD / 64 slabs of 64 columns.
template <int HD>
struct Lay {
  static_assert(HD == 64 || HD == 128, "head dimension");
  static constexpr int SLABS = HD / 64;
  static constexpr int SM_K = 0;
  static constexpr int SM_V = SM_K + SLABS * KSLAB;
  static constexpr int SM_STAGE = SM_V + SLABS * KSLAB;
  static constexpr int STAGE_BYTES = 2 * SLABS * QSLAB;     // Q_i + dO_i
  static constexpr int SM_DS = SM_STAGE + NS * STAGE_BYTES; // dS^T [128 keys][128 queries] bf16, 2 slabs
  static constexpr int SM_BIG = SM_DS + 2 * KSLAB;          // end of the operand block
  static constexpr uint32_t ID_GRAD = idesc(BK, HD, 0, 1);  // dV, dK: P^T (TMEM) / dS^T (smem, K-major), dO / Q MN-major
  static constexpr uint32_t ID_DQ = idesc(BQ, HD, 1, 1);    // dQ: dS (from dS^T) and K, both MN-major
  static_assert(SM_BIG + 1023 + NS * VEC_BYTES <= SMEM_ALLOC, "operand block + vectors, small block in front");
  static_assert(SM_BIG + SMALL_BYTES - 1 + SMALL_BYTES + NS * VEC_BYTES <= SMEM_ALLOC, "everything behind");
  // the dQ of a step, staged as fp32 32 x 32 boxes (HD / 32 per lane quarter), fits a finished stage
  static_assert(4 * (HD / 32) * 32 * 128 <= STAGE_BYTES, "dQ staging");
};

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off16) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(d));
  lo += off16;
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kAttnWaitNs) break;
  }
}

struct BwdParams {
  const float* nlse2;  // [B*Hq][Nq_pad]: -LSE * log2(e); -inf on padding and on rows with no key
                       // (Nq_pad: Nq rounded up to 128)
  const float* ndelta; // [B*Hq][Nq_pad]: -scale * rowsum(dO * O); 0 on padding
  float* dq;           // [B, Hq, Nq, D] fp32, accumulated (zeroed before the launch)
  __nv_bfloat16* dk;   // [B, Hkv, Nk, D]
  __nv_bfloat16* dv;
  int B, Hq, Hkv, Nq, Nk, Nq_pad, group;
  float c_log2;        // scale * log2(e)
  float scale;
  int causal;
  int window;          // > 0: key k visible to query q only if k > q + Nk - Nq - window
  int* err;
};

// -scale * D (D = rowsum(dO * O)) and -LSE * log2(e) per query row, padded to
// 128 rows per head, negated so that the main kernel needs one fused
// multiply-add per score.
template <int HD>
__global__ void __launch_bounds__(256)
attn_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                     const float* __restrict__ lse, float* __restrict__ nlse2, float* __restrict__ ndelta,
                     long long rows_pad, int Nq, int Nq_pad, float scale) {
  const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  if (r >= rows_pad) return;
  const long long bh = r / Nq_pad;
  const int i = static_cast<int>(r - bh * Nq_pad);
  if (i >= Nq) {
    if (lane == 0) {
      ndelta[r] = 0.f;
      nlse2[r] = -CUDART_INF_F;
    }
    return;
  }
  float s;
  if constexpr (HD == 128) {   // four elements per lane
    const long long src = (bh * Nq + i) * HD + lane * 4;
    const uint2 uo = *reinterpret_cast<const uint2*>(o + src);
    const uint2 ud = *reinterpret_cast<const uint2*>(dout + src);
    const float o4[4] = {__uint_as_float(uo.x << 16), __uint_as_float(uo.x & 0xFFFF0000u),
                         __uint_as_float(uo.y << 16), __uint_as_float(uo.y & 0xFFFF0000u)};
    const float d4[4] = {__uint_as_float(ud.x << 16), __uint_as_float(ud.x & 0xFFFF0000u),
                         __uint_as_float(ud.y << 16), __uint_as_float(ud.y & 0xFFFF0000u)};
    s = (o4[0] * d4[0] + o4[1] * d4[1]) + (o4[2] * d4[2] + o4[3] * d4[3]);
  } else {                     // two elements per lane
    const long long src = (bh * Nq + i) * HD + lane * 2;
    const uint32_t uo = *reinterpret_cast<const uint32_t*>(o + src);
    const uint32_t ud = *reinterpret_cast<const uint32_t*>(dout + src);
    s = __uint_as_float(uo << 16) * __uint_as_float(ud << 16) +
        __uint_as_float(uo & 0xFFFF0000u) * __uint_as_float(ud & 0xFFFF0000u);
  }
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
  if (lane == 0) {
    ndelta[r] = -scale * s;
    const float l = lse[bh * Nq + i];
    nlse2[r] = l == -CUDART_INF_F ? -CUDART_INF_F : -l * 1.4426950408889634f;
  }
}

template <int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using LY = Lay<HD>;
  constexpr int SLABS = LY::SLABS;
  constexpr int SM_K = LY::SM_K, SM_V = LY::SM_V, SM_STAGE = LY::SM_STAGE, STAGE_BYTES = LY::STAGE_BYTES;
  constexpr int SM_DS = LY::SM_DS, SM_BIG = LY::SM_BIG;
  constexpr uint32_t ID_GRAD = LY::ID_GRAD, ID_DQ = LY::ID_DQ;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = smem_u32(smem);
  const bool small_front = pad >= static_cast<uint32_t>(SMALL_BYTES);
  uint8_t* small = small_front ? smem_raw : smem + SM_BIG;
  const uint32_t sbar = smem_u32(small);
  uint8_t* vecs = smem + SM_BIG + (small_front ? 0 : SMALL_BYTES);  // per stage: -LSE*log2(e), -scale*D
  const uint32_t svec = smem_u32(vecs);
  const int warp = warp_id_uniform();
  const int lane = static_cast<int>(lane_id());

  const uint32_t bar_kv_full = sbar;                                        // K_j, V_j landed
  auto bar_q_full = [&](int s) { return sbar + 8u * (1 + s); };              // stage s landed
  auto bar_q_empty = [&](int s) { return sbar + 8u * (1 + NS + s); };        // stage s read by every MMA and
                                                                            // by the dQ reduce copies
  const uint32_t bar_s_full = sbar + 8u * (1 + 2 * NS);                     // S^T in TMEM
  const uint32_t bar_p_ready = bar_s_full + 8;                              // P^T written
  const uint32_t bar_dp_full = bar_s_full + 16;                             // dP^T in TMEM
  const uint32_t bar_ds_ready = bar_s_full + 24;                            // dS^T written
  const uint32_t bar_dq_full = bar_s_full + 32;                             // dQ in TMEM
  const uint32_t bar_dq_empty = bar_s_full + 40;                            // dQ read out
  const uint32_t bar_kv_done = bar_s_full + 48;                             // dK, dV complete
  const uint32_t bar_mma_done = bar_s_full + 56;                            // every MMA complete
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(small + NUM_BARS * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + NUM_BARS * 8 + 4);

  const int j0 = static_cast<int>(blockIdx.x) * BK;
  const int kvh = static_cast<int>(blockIdx.y);
  const int b = static_cast<int>(blockIdx.z);
  const int off = p.Nk - p.Nq;  // bottom-right causal: key k visible to query q iff k <= q + off
  const int n_qt = (p.Nq + BQ - 1) / BQ;
  int it0 = 0;  // first query tile with a query that sees a key of this tile
  if (p.causal && j0 - off > 0) it0 = (j0 - off) / BQ;
  // sliding window: key k is visible to query q only if q < k - off + window, so the
  // tile's last key (j0 + BK - 1) bounds the last query tile
  int it_end = n_qt;
  if (p.window > 0) {
    const long long q_last = static_cast<long long>(j0) + BK - 1 - off + p.window - 1;
    it_end = q_last < 0 ? 0 : static_cast<int>(min(static_cast<long long>(n_qt), q_last / BQ + 1));
  }
  const int per_head = max(0, it_end - it0);
  const int n_steps = per_head * p.group;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_q_full(s), 1);
      mbar_init(bar_q_empty(s), 1 + 4);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_p_ready, NROW);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_ds_ready, NROW);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_empty, 4);
    mbar_init(bar_kv_done, 1);
    mbar_init(bar_mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Each CTA walks its query tiles from a different start (rotated by its key
  // tile): the CTAs of one head then add into different dQ rows at any moment
  // instead of all into the same ones, which the L2 would serialise.
  const int rot = per_head > 0 ? static_cast<int>(blockIdx.x) % per_head : 0;
  auto step_head = [&](int step) { return kvh * p.group + step / max(per_head, 1); };
  auto step_q0 = [&](int step) {
    int t = step % max(per_head, 1) + rot;
    if (t >= per_head) t -= per_head;
    return (it0 + t) * BQ;
  };

  if (warp == WARP_TMA) {
    // ================================================================ producer
    if (lane == 0 && n_steps > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar_kv_full, 2 * SLABS * KSLAB);
      for (int kb = 0; kb < SLABS; ++kb) {
        tma_load_3d(sb + SM_K + kb * KSLAB, &tm_k, bar_kv_full, kb * 64, j0, b * p.Hkv + kvh);
        tma_load_3d(sb + SM_V + kb * KSLAB, &tm_v, bar_kv_full, kb * 64, j0, b * p.Hkv + kvh);
      }
      int step = 0;
      bool ok = true;
      for (; step < n_steps && ok; ++step) {
        const int s = step % NS, use = step / NS;
        if (use > 0 && !mbar_wait(bar_q_empty(s), (use - 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const int h = step_head(step), i0 = step_q0(step);
        const uint32_t st = sb + SM_STAGE + s * STAGE_BYTES;
        const uint32_t vec = svec + s * VEC_BYTES;
        mbar_arrive_expect_tx(bar_q_full(s), STAGE_BYTES + VEC_BYTES);
        for (int kb = 0; kb < SLABS; ++kb) {
          tma_load_3d(st + kb * QSLAB, &tm_q, bar_q_full(s), kb * 64, i0, b * p.Hq + h);
          tma_load_3d(st + SLABS * QSLAB + kb * QSLAB, &tm_do, bar_q_full(s), kb * 64, i0, b * p.Hq + h);
        }
        const size_t vrow = (static_cast<size_t>(b) * p.Hq + h) * p.Nq_pad + i0;
        bulk_load(vec, p.nlse2 + vrow, BQ * 4, bar_q_full(s));
        bulk_load(vec + BQ * 4, p.ndelta + vrow, BQ * 4, bar_q_full(s));
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        drain_wait(bar_kv_full, 0);
        for (int i = max(0, step - NS); i < step; ++i) drain_wait(bar_q_full(i % NS), (i / NS) & 1);
      }
    }
  } else if (warp == WARP_MMA) {
    // ================================================================ MMA issuer
    if (lane == 0 && n_steps > 0) {
      const uint64_t k_kmaj = smem_desc_sw128(sb + SM_K, 16, 1024);   // K as A, K-major
      const uint64_t v_kmaj = smem_desc_sw128(sb + SM_V, 16, 1024);
      const uint64_t k_mn = smem_desc_sw128(sb + SM_K, KSLAB, 1024);  // K as B, MN-major
      const uint64_t ds_mn = smem_desc_sw128(sb + SM_DS, KSLAB, 1024); // dS (stored as dS^T) as A, MN-major
      const uint64_t ds_kmaj = smem_desc_sw128(sb + SM_DS, 16, 1024);  // dS^T as A, K-major
      bool ok = mbar_wait(bar_kv_full, 0, abort_flag, p.err);
      for (int step = 0; step < n_steps && ok; ++step) {
        const int s = step % NS;
        const uint32_t st = sb + SM_STAGE + s * STAGE_BYTES;
        const uint64_t q_kmaj = smem_desc_sw128(st, 16, 1024);
        const uint64_t do_kmaj = smem_desc_sw128(st + SLABS * QSLAB, 16, 1024);
        const uint64_t q_mn = smem_desc_sw128(st, QSLAB, 1024);
        const uint64_t do_mn = smem_desc_sw128(st + SLABS * QSLAB, QSLAB, 1024);
        if (!mbar_wait(bar_q_full(s), (step / NS) & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        // S^T = K_j Q_i^T (over P^T of the previous step: the dV MMA that read it came first)
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t a_off = static_cast<uint32_t>((kk >> 2) * KSLAB + (kk & 3) * 32) >> 4;
          const uint32_t b_off = static_cast<uint32_t>((kk >> 2) * QSLAB + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + COL_S, desc_add(k_kmaj, a_off), desc_add(q_kmaj, b_off), ID_ST, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_s_full);
        // dP^T = V_j dO_i^T over the previous step's dQ: it must have been read out
        if (step > 0 && !mbar_wait(bar_dq_empty, (step - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t a_off = static_cast<uint32_t>((kk >> 2) * KSLAB + (kk & 3) * 32) >> 4;
          const uint32_t b_off = static_cast<uint32_t>((kk >> 2) * QSLAB + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + COL_DP, desc_add(v_kmaj, a_off), desc_add(do_kmaj, b_off), ID_ST, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_dp_full);
        // dV_j += P^T dO_i (16 queries per K step)
        if (!mbar_wait(bar_p_ready, step & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          // P^T of queries [64 hf, +64) sits in columns [64 hf, +32) (bf16 pairs)
          const uint32_t a_col = COL_S + (kk >> 2) * 64 + (kk & 3) * 8;
          const uint32_t boff = static_cast<uint32_t>(kk * 16 * 128) >> 4;
          mma_bf16_ts(tmem + COL_DV, tmem + a_col, desc_add(do_mn, boff), ID_GRAD, (step > 0 || kk > 0) ? 1u : 0u);
        }
        // dK_j += dS^T Q_i
        if (!mbar_wait(bar_ds_ready, step & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t a_off = static_cast<uint32_t>((kk >> 2) * KSLAB + (kk & 3) * 32) >> 4;
          const uint32_t boff = static_cast<uint32_t>(kk * 16 * 128) >> 4;
          mma_bf16_ss(tmem + COL_DK, desc_add(ds_kmaj, a_off), desc_add(q_mn, boff), ID_GRAD,
                      (step > 0 || kk > 0) ? 1u : 0u);
        }
        // dQ_i = dS K_j (16 keys per K step), over dP^T (read by the row warps before ds_ready)
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint32_t off16 = static_cast<uint32_t>(kk * 16 * 128) >> 4;
          mma_bf16_ss(tmem + COL_DQ, desc_add(ds_mn, off16), desc_add(k_mn, off16), ID_DQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_dq_full);
        mma_commit(bar_q_empty(s));
      }
      if (ok) mma_commit(bar_kv_done);
      mma_commit(bar_mma_done);
      drain_wait(bar_mma_done, 0);
    }
  } else {
    // ================================================================ row warps (0..7), dQ warps (10..13)
    const bool dq_warp = warp >= WARP_DQ0;
    const int quad = warp & 3;
    const int hf = dq_warp ? 0 : warp >> 2;  // query half of a row warp
    const uint32_t lane_sel = static_cast<uint32_t>(quad * 32) << 16;
    const int r = quad * 32 + lane;  // key row (S^T, dP^T, dV, dK) / query row (dQ) of this thread
    const int key = j0 + r;
    const bool key_ok = key < p.Nk;
    bool ok = true;
    for (int step = 0; step < n_steps && ok; ++step) {
      const int s = step % NS;
      const int h = step_head(step), i0 = step_q0(step);
      if (dq_warp) {
        // dQ_i: this thread holds query r of the step.  Stage it in the
        // finished Q/dO stage (its MMAs are complete: dq_full follows them) as
        // four 32-query x 32-dim boxes per warp, 128-byte rows with the
        // 128-byte swizzle (16-byte chunk c of row l at chunk c ^ (l % 8)).
        ok = __all_sync(0xffffffffu, mbar_wait(bar_dq_full, step & 1, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        uint8_t* box0 = smem + SM_STAGE + s * STAGE_BYTES + quad * ((HD / 32) * 32 * 128);
#pragma unroll
        for (int hh = 0; hh < HD / 64; ++hh) {
          uint32_t qr[2][32];
          tmem_ld32(tmem + lane_sel + COL_DQ + 64 * hh, qr[0]);
          tmem_ld32(tmem + lane_sel + COL_DQ + 64 * hh + 32, qr[1]);
          tmem_wait_ld();
          if (hh == HD / 64 - 1) {  // the columns are free for the next dP^T
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dq_empty);
          }
#pragma unroll
          for (int bx = 0; bx < 2; ++bx)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(box0 + (2 * hh + bx) * (32 * 128) + lane * 128 + ((c ^ (lane & 7)) * 16)) =
                  make_uint4(qr[bx][4 * c], qr[bx][4 * c + 1], qr[bx][4 * c + 2], qr[bx][4 * c + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // rows past the sequence end fall outside the map and are skipped
          if (i0 + quad * 32 < p.Nq) {
#pragma unroll
            for (int bx = 0; bx < HD / 32; ++bx)
              tma_reduce_add_3d(&tm_dq, smem_u32(box0 + bx * (32 * 128)), bx * 32, i0 + quad * 32, b * p.Hq + h);
          }
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(bar_q_empty(s));  // the stage may be refilled
        }
        __syncwarp();
        continue;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar_q_full(s), (step / NS) & 1, abort_flag, p.err) &&
                                       mbar_wait(bar_s_full, step & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const float* nlse2v = reinterpret_cast<const float*>(vecs + s * VEC_BYTES) + 64 * hf;
      const float* ndeltav = reinterpret_cast<const float*>(vecs + s * VEC_BYTES) + BQ + 64 * hf;
      // causal: query c of this step sees this key iff key <= i0 + c + off; window: iff
      // i0 + c < key - off + window
      const int c_min = p.causal ? key - off - i0 - 64 * hf : 0;  // first visible query of this half
      const int c_max = p.window > 0 ? key - off + p.window - 1 - i0 - 64 * hf : 63;  // last visible
      // P^T = 2^(S^T scale log2(e) - LSE log2(e)) for queries [64 hf, +64),
      // packed as bf16 pairs into S^T columns [64 hf, +32) (read by this warp only)
      {
        uint32_t sr[2][32];
        tmem_ld32(tmem + lane_sel + COL_S + 64 * hf, sr[0]);
        tmem_ld32(tmem + lane_sel + COL_S + 64 * hf + 32, sr[1]);
        tmem_wait_ld();
        const uint64_t c_log2_2 = f2_pack(p.c_log2, p.c_log2);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(nlse2v + c);  // one broadcast load
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int cl = c + e;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[cl >> 5][cl & 31]), __uint_as_float(sr[cl >> 5][(cl & 31) + 1])),
                             c_log2_2, e == 0 ? f2_pack(l4.x, l4.y) : f2_pack(l4.z, l4.w)),
                      x0, x1);
            pk[cl >> 1] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
          }
        }
        // masked entries (padding keys, causal, window) to 0: only warps that have some
        if (!__all_sync(0xffffffffu, key_ok && c_min <= 0 && c_max >= 63)) {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const bool v0 = key_ok && c >= c_min && c <= c_max, v1 = key_ok && c + 1 >= c_min && c + 1 <= c_max;
            pk[c >> 1] &= (v0 ? 0x0000FFFFu : 0u) | (v1 ? 0xFFFF0000u : 0u);
          }
        }
        tmem_st32(tmem + lane_sel + COL_S + 64 * hf, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_ready);
      // dS^T = P^T (scale dP^T - scale D) for queries [64 hf, +64), 32 at a
      // time, from the packed P^T, as bf16 into row r of shared-memory slab hf
      // (128-byte rows, 128-byte swizzle: 16-byte chunk c of a row sits at
      // chunk c ^ (r % 8)).  The previous step's dK and dQ MMAs have read that
      // tile: they completed before dP^T.
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dp_full, step & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      {
        const uint64_t scale2 = f2_pack(p.scale, p.scale);
        uint8_t* ds_row = smem + SM_DS + hf * KSLAB + r * 128;
#pragma unroll
        for (int qc = 0; qc < 2; ++qc) {
          uint32_t dr[32], pp[16];
          tmem_ld32(tmem + lane_sel + COL_DP + 64 * hf + 32 * qc, dr);
          tmem_ld16(tmem + lane_sel + COL_S + 64 * hf + 16 * qc, pp);
          tmem_wait_ld();
          uint32_t dk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(ndeltav + 32 * qc + c);  // one broadcast load
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const int cl = c + e;
              const uint64_t p2 =
                  f2_pack(__uint_as_float(pp[cl >> 1] << 16), __uint_as_float(pp[cl >> 1] & 0xFFFF0000u));
              const uint64_t dp2 = f2_pack(__uint_as_float(dr[cl]), __uint_as_float(dr[cl + 1]));
              float d0, d1;
              f2_unpack(f2_mul(p2, f2_fma(dp2, scale2, e == 0 ? f2_pack(d4.x, d4.y) : f2_pack(d4.z, d4.w))), d0, d1);
              dk[cl >> 1] = pack_bf16x2(d0, d1);
            }
          }
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            *reinterpret_cast<uint4*>(ds_row + (((4 * qc + c4) ^ (r & 7)) * 16)) =
                make_uint4(dk[4 * c4], dk[4 * c4 + 1], dk[4 * c4 + 2], dk[4 * c4 + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds_ready);
    }
    if (dq_warp && lane == 0) bulk_wait_group0();  // the dQ adds are complete before the CTA exits
    // dV_j (row warps of query half 0) or dK_j (row warps of query half 1): this thread's key row
    if (ok && !dq_warp) {
      if (n_steps > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar_kv_done, 0, abort_flag, p.err));
      if (ok) {
        tc_fence_after();
        const size_t orow = (static_cast<size_t>(b) * p.Hkv + kvh) * p.Nk + key;
        uint4* dst = reinterpret_cast<uint4*>((hf ? p.dk : p.dv) + orow * HD);
#pragma unroll
        for (int ch = 0; ch < HD / 32; ++ch) {
          uint32_t g[32];
          if (n_steps > 0) {
            tmem_ld32(tmem + lane_sel + (hf ? COL_DK : COL_DV) + ch * 32, g);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = 0u;
          }
          if (key_ok) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[4 * ch + i] = make_uint4(pack_bf16x2(__uint_as_float(g[8 * i + 0]), __uint_as_float(g[8 * i + 1])),
                                           pack_bf16x2(__uint_as_float(g[8 * i + 2]), __uint_as_float(g[8 * i + 3])),
                                           pack_bf16x2(__uint_as_float(g[8 * i + 4]), __uint_as_float(g[8 * i + 5])),
                                           pack_bf16x2(__uint_as_float(g[8 * i + 6]), __uint_as_float(g[8 * i + 7])));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace bwd

size_t bwd_workspace_bytes(int B, int Hq, int Nq) {
  const size_t nq_pad = static_cast<size_t>((Nq + bwd::BQ - 1) / bwd::BQ) * bwd::BQ;
  return 2 * static_cast<size_t>(B) * Hq * nq_pad * sizeof(float);
}

namespace bwd {

template <int HD>
int launch_bwd_hd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, float* dq, void* dk, void* dv, void* workspace, int B, int Hq,
                  int Hkv, int Nq, int Nk, float scale, int causal, int window, cudaStream_t stream,
                  int* err) {
  const int nq_pad = (Nq + BQ - 1) / BQ * BQ;
  const long long rows_pad = static_cast<long long>(B) * Hq * nq_pad;
  float* nlse2 = static_cast<float*>(workspace);
  float* ndelta = nlse2 + rows_pad;
  if (cudaMemsetAsync(dq, 0, static_cast<size_t>(B) * Hq * Nq * HD * sizeof(float), stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  attn_bwd_prep_kernel<HD><<<static_cast<unsigned>((rows_pad + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, nlse2, ndelta,
      rows_pad, Nq, nq_pad, scale);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo, tdq;
  const uint32_t box_q[3] = {64, BQ, 1};
  const uint32_t box_k[3] = {64, BK, 1};
  const uint32_t box_dq[3] = {32, 32, 1};
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_tiled_3d(&tq, dt, q, HD, Nq, static_cast<uint64_t>(B) * Hq, 2, box_q, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tdo, dt, dout, HD, Nq, static_cast<uint64_t>(B) * Hq, 2, box_q, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tk, dt, k, HD, Nk, static_cast<uint64_t>(B) * Hkv, 2, box_k, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tv, dt, v, HD, Nk, static_cast<uint64_t>(B) * Hkv, 2, box_k, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dq, HD, Nq, static_cast<uint64_t>(B) * Hq, 4, box_dq,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return ATTN_ERR_CUDA;
  static KernelSetup setup;
  if (const int rc = prepare_kernel(setup, attn_bwd_kernel<HD>, SMEM_ALLOC); rc != ATTN_OK) return rc;
  BwdParams prm;
  prm.nlse2 = nlse2;
  prm.ndelta = ndelta;
  prm.dq = dq;
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.Nq_pad = nq_pad;
  prm.group = Hq / Hkv;
  prm.c_log2 = scale * 1.4426950408889634f;
  prm.scale = scale;
  prm.causal = causal ? 1 : 0;
  prm.window = window > 0 ? window : 0;
  prm.err = err;
  const dim3 grid((Nk + BK - 1) / BK, Hkv, B);
  attn_bwd_kernel<HD><<<grid, NTHREADS, SMEM_ALLOC, stream>>>(tq, tk, tv, tdo, tdq, prm);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace bwd

int launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
               const float* lse, float* dq, void* dk, void* dv, void* workspace, int B, int Hq,
               int Hkv, int Nq, int Nk, int D, float scale, int causal, int window, cudaStream_t stream,
               int* err) {
  if (D == 128)
    return bwd::launch_bwd_hd<128>(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, Hq, Hkv, Nq, Nk, scale,
                                   causal, window, stream, err);
  if (D == 64)
    return bwd::launch_bwd_hd<64>(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, Hq, Hkv, Nq, Nk, scale,
                                  causal, window, stream, err);
  return ATTN_ERR_HEAD_DIM;
}

}  // namespace attn

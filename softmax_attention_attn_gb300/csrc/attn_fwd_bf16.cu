// attn_fwd_bf16.cu — bf16 / fp16 fused attention forward for sm_103a on tcgen05.
//
// What it computes (softmax attention, "Agent 帮我写 CUDA：一个 Softmax Attention
// 算子的开发全记录" section 二 "参考基线"; online softmax over K/V tiles, same page
// section 四 "Tiled Attention 的核心思想"; GQA / causal / sliding window from
// "Ask, Don't Equip: ..." section "研究动机"):
//   O = softmax(scale * Q K^T + mask) V,  LSE = ln sum_j exp(scale * q.k_j)
// The three-stage split (QK matmul, row softmax, PV matmul) is the tile
// decomposition of the PTO FlashAttention article's section "为什么 PTO 适合
// Agent 来优化"; here each stage is mapped onto Blackwell hardware:
//
//   * persistent CTAs (one per SM) walk a list of work units — two 128-row Q
//     tiles of one (batch, head); causal lists put the longest units first and
//     passes over the list alternate the direction in which units are dealt
//     to the CTAs — and stream 128-key K/V tiles through a TMA ring (4 slots at
//     D = 128; 128-byte swizzle, mbarrier transaction counts).  Three Q tile
//     buffers rotate over the units' Q tiles, so the next unit's Q lands while
//     the current one runs.  Barriers and tensor memory are set up once; the
//     next unit's Q, K/V and first S overlap the last unit's epilogue;
//   * 512 threads in four warpgroups, each given its register share by setmaxnreg
//     (the softmax warpgroups take more than the 128 a thread is launched with);
//   * warps 0-3 and 4-7 are the softmax warps of Q tile 0 and 1: warp w
//     reaches tensor-memory lanes 32 (w % 4) .. + 31, so thread r of warp w
//     owns row 32 (w % 4) + r; it loads its 128 scores, applies the mask,
//     updates the running max / sum in the exp2 domain, rescales its O row in
//     tensor memory when the max grew by more than 2^8 (otherwise the stale max
//     is kept; the final normalisation is exact either way), writes P as bf16
//     over its S columns and signals its MMA issuer; at the end of a unit it
//     writes LSE and hands 1 / l to the epilogue warps through shared memory;
//   * warps 8-11 are the epilogue: once a unit's last P V has completed they
//     read O out of tensor memory, hand it back to the MMA issuer, divide by
//     the row sum, round to bf16 and write O (32-byte stores when O is 32-byte
//     aligned), while the softmax warps already run the next unit;
//   * warps 12 and 13 issue the tcgen05.mma of Q tile 0 and 1 (lane 0 of a
//     converged warp): S_t = Q_t K^T into tensor memory (fp32, 128 columns per
//     Q tile), then O_t += P_t V with P read from tensor memory (the TS form)
//     and V from shared memory (MN-major operand); the two take strict turns,
//     one key tile at a time, and wait and commit outside their turn;
//   * warp 14 (one elected thread) is the TMA producer, with L2 policies: Q
//     evict-first (read once), K/V evict-last (read by every q-block of a head);
//     warp 15 only completes the last warpgroup;
//   * with QK8, Q and K are E4M3 codes and S = Q K^T runs on kind::f8f6f4
//     (the fp8 prefill; V arrives widened to bf16).
//
// The two Q tiles ping-pong: while the softmax warps of tile 0 work on tile j the
// tensor core computes PV_1(j-1) and S_1(j), and vice versa.
//
// Tensor memory (512 columns): S_0 [0,128) S_1 [128,256) O_0 [256,384) O_1 [384,512);
// P_t aliases the first 64 columns of S_t (two bf16 per 32-bit column).
#include <cuda_runtime.h>
#include <math_constants.h>

#include <atomic>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace fwd_bf16 {

constexpr int BM = 128;                      // query rows per Q tile
constexpr int BN = 128;                      // keys per K/V tile
constexpr int NQT = 2;                       // Q tiles per work unit
constexpr int KBLK_BYTES = 128 * 64 * 2;     // 64-column (128-byte) slab of a 128-row tile
constexpr int NUM_SOFTMAX_WARPS = 4 * NQT;
constexpr int WARP_SOFTMAX0 = 0;                     // softmax warps of Q tile t: WARP_SOFTMAX0 + 4t ..
constexpr int WARP_EPI = NUM_SOFTMAX_WARPS;          // epilogue warps: WARP_EPI + q reads TMEM lanes 32q ..
constexpr int WARP_MMA = WARP_EPI + 4;               // issuer of Q tile t is warp WARP_MMA + t
constexpr int WARP_TMA = WARP_MMA + NQT;             // TMA producer (the warp after it idles)
constexpr int NTHREADS = (WARP_TMA + 2) * 32;        // four warpgroups
// Registers per thread after each warpgroup's setmaxnreg: the block is launched with
// 65536 / NTHREADS = 128 each; the two softmax warpgroups take more, the epilogue and
// control (issuers, TMA) warpgroups give theirs up, and the shares add up to the block's
// (an `inc` beyond the pool would wait forever).  The epilogue holds a packed output
// row (HD / 2 words) and one 32-column piece of O.
template <int HD, bool CAP>
struct Regs {
  static constexpr int SOFTMAX = (HD == 64 || CAP) ? 176 : 168;
  static constexpr int CTRL = CAP ? 56 : 72;
  static constexpr int EPI = (65536 - 2 * 128 * SOFTMAX - 128 * CTRL) / 128;
  static_assert(2 * 128 * SOFTMAX + 128 * EPI + 128 * CTRL == 65536 && EPI % 8 == 0, "register shares");
};
static_assert(NTHREADS == 512 && NUM_SOFTMAX_WARPS == 8, "four warpgroups: softmax x2, epilogue, control");
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;         // keep a stale max while the growth is <= 2^8

// Shape constants for head dimension HD (64 or 128); F16 selects fp16 instead
// of bf16 operands; QK8 selects E4M3 Q and K (S = Q K^T on kind::f8f6f4; V, P
// and O stay bf16).
template <int HD, bool F16 = false, bool QK8 = false>
struct Cfg {
  static constexpr int KBLKS = HD / 64;                 // 128-byte slabs per 16-bit tile row
  static constexpr int TILE_BYTES = KBLKS * KBLK_BYTES; // one 128-row 16-bit tile (a ring slot)
  static constexpr int QK_BOX = QK8 ? 128 : 64;         // Q/K elements per 128-byte slab row
  static constexpr int QK_SLABS = HD / QK_BOX;          // 128-byte slabs per Q/K tile row
  static constexpr int QK_TILE_BYTES = QK_SLABS * KBLK_BYTES;  // one 128-row Q or K tile
  static constexpr int QK_STEPS = QK8 ? HD / 32 : HD / 16;     // MMAs of one Q K^T (32 bytes of K each)
  static constexpr int STAGES = HD == 128 ? (QK8 ? 5 : 4) : 10;  // K/V ring slots (one K or V tile each)
  // Q tile buffers: three rotate over the Q tiles of successive units (tile t of the
  // n-th unit with work in buffer (2n + t) % 3), so the next unit's Q tile 0 loads
  // while the current unit runs and its Q tile 1 as soon as the current tile 0 is done
  static constexpr int NQB = 3;
  static constexpr int SMEM_Q = 0;
  static constexpr int SMEM_RING = SMEM_Q + NQB * QK_TILE_BYTES;
  static constexpr int SMEM_BAR = SMEM_RING + STAGES * TILE_BYTES;
  static constexpr int NUM_BARS = 2 * NQB + 1 + 2 * STAGES + 7 * NQT;
  static constexpr int SMEM_MISC = SMEM_BAR + NUM_BARS * 8;
  static constexpr int SMEM_STATS = SMEM_MISC + 16;     // per Q tile row: 1 / l for the epilogue warps
  static constexpr int SMEM_ALLOC = SMEM_STATS + NQT * BM * 4 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t AB_FORMAT = F16 ? 0u : 1u;  // instruction-descriptor A/B format
  static constexpr uint32_t IDESC_QK = QK8 ? idesc_e4m3_f32(128, BN) : idesc_f16kind_f32(128, BN, 0, AB_FORMAT);
  static constexpr uint32_t IDESC_PV = idesc_f16kind_f32(128, HD, 1, AB_FORMAT);
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
  static_assert(2 * BN + 2 * HD <= TMEM_COLS, "tensor memory budget");
  static_assert(!QK8 || (HD == 128 && !F16), "E4M3 Q/K: bf16 V/O and HD = 128 only");
};

// Softcap fast paths: tanh(y) ~= y * sum_k t_k y^(2k), minimax polynomials of the same
// accuracy (largest relative error 5.4e-7 / 5.9e-7; 5.9e-7 / 6.7e-7 evaluated in fp32 by
// Horner's rule) on |y| <= 0.5 (short) and |y| <= 1 (long), found by the Remez exchange in
// softmax_attention_attn_gb300/tanh_fit.py.
constexpr double kTanhPolyShort[4] = {0.99999945577093852, -0.3332631793594138, 0.1319029660321,
                                      -0.044402226127707133};
constexpr double kTanhPolyShortYMax = 0.5;
constexpr double kTanhPolyLong[6] = {0.99999941359925792, -0.33329042378530915, 0.13281433880740096,
                                     -0.051605674002214393, 0.016743115063837057, -0.003067060326585761};
constexpr double kTanhPolyLongYMax = 1.0;

// In place: s[i] <- s[i] * P(s[i]^2) with P(w) = sum_k coef[k] w^k (Horner's rule on
// f32x2 pairs); *rmax <- the same for the scalar *rmax.
template <int TERMS, int N>
__device__ __forceinline__ void cap_polynomial(float (&s)[N], float* rmax, const float* coef) {
  uint64_t cf[TERMS];
#pragma unroll
  for (int k = 0; k < TERMS; ++k) cf[k] = f2_pack(coef[k], coef[k]);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const uint64_t s2 = f2_pack(s[i], s[i + 1]);
    const uint64_t w2 = f2_mul(s2, s2);
    uint64_t q2 = f2_fma(cf[TERMS - 1], w2, cf[TERMS - 2]);
#pragma unroll
    for (int k = TERMS - 3; k >= 0; --k) q2 = f2_fma(q2, w2, cf[k]);
    f2_unpack(f2_mul(s2, q2), s[i], s[i + 1]);
  }
  const float w = *rmax * *rmax;
  float q = fmaf(coef[TERMS - 1], w, coef[TERMS - 2]);
#pragma unroll
  for (int k = TERMS - 3; k >= 0; --k) q = fmaf(q, w, coef[k]);
  *rmax *= q;
}

__device__ __forceinline__ uint32_t s_col(int t) { return static_cast<uint32_t>(t * BN); }
template <int HD>
__device__ __forceinline__ uint32_t o_col(int t) { return static_cast<uint32_t>(NQT * BN + t * HD); }

// Two floats -> one 32-bit pair of the operand type (bf16 or fp16), RNE.
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

// tanh from the exponential: tanh|y| = 1 - 2 / (1 + e^(2|y|)), sign restored
// (hardware 2^x and 1/x; e^(2|y|) = inf gives 1).  Its absolute error stays
// near one fp32 ulp of 1, including for small |y|.
__device__ __forceinline__ float tanh_exp(float y) {
  const float e = ex2_approx(fabsf(y) * 2.8853900817779268f);  // 2^(2|y| log2 e)
  return copysignf(fmaf(-2.f, rcp_approx(1.f + e), 1.f), y);
}

// Shared-memory descriptors are linear in the start address (its field is
// address >> 4 in the low 14 bits, and every shared-memory address here is
// below 2^18), so a descriptor for base + offset is the base descriptor plus
// offset >> 4 in its low word.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off16) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(d));
  lo += off16;
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

// S (tmem) = Q_tile (smem) x K_tile^T (smem); both K-major, 128-byte swizzle,
// given by the descriptors of their first byte.  Every MMA takes 32 bytes of
// each row (16 bf16 / fp16 or 32 E4M3 elements), four per 128-byte slab.
template <int HD, bool F16, bool QK8>
__device__ __forceinline__ void issue_qk(uint32_t issue, uint32_t d_tmem, uint64_t q_desc,
                                         uint64_t k_desc) {
  using C = Cfg<HD, F16, QK8>;
#pragma unroll
  for (int kk = 0; kk < C::QK_STEPS; ++kk) {
    const uint32_t koff = static_cast<uint32_t>((kk >> 2) * KBLK_BYTES + (kk & 3) * 32) >> 4;
    if constexpr (QK8)
      mma_f8_ss_if(issue, d_tmem, desc_add(q_desc, koff), desc_add(k_desc, koff), C::IDESC_QK,
                   kk > 0 ? 1u : 0u);
    else
      mma_bf16_ss_if(issue, d_tmem, desc_add(q_desc, koff), desc_add(k_desc, koff), C::IDESC_QK,
                     kk > 0 ? 1u : 0u);
  }
}

// O (tmem) (+)= P (tmem, bf16) x V_tile (smem, MN-major: d contiguous), for the
// 16-key steps kk in [kk0, kk0 + 4): one half of the tile's keys.  With HD =
// 128 the two 64-column slabs of V are KBLK_BYTES apart (the leading byte
// offset of the MN-major operand, part of v_desc); with HD = 64 there is one slab.
template <int HD, bool F16>
__device__ __forceinline__ void issue_pv_half(uint32_t issue, uint32_t d_tmem, uint32_t p_tmem,
                                              uint64_t v_desc, bool accumulate, int kk0) {
#pragma unroll
  for (int kk = kk0; kk < kk0 + BN / 32; ++kk) {
    mma_bf16_ts_if(issue, d_tmem, p_tmem + static_cast<uint32_t>(kk * 8),
                desc_add(v_desc, static_cast<uint32_t>(kk * 16 * 128) >> 4), Cfg<HD, F16>::IDESC_PV,
                (accumulate || kk > 0) ? 1u : 0u);
  }
}

// A position in the K/V ring: slot and the parity of its fill / release phase.
struct RingPos {
  int slot;
  uint32_t phase;
};
template <int STAGES>
__device__ __forceinline__ RingPos ring_pos(int pos) {
  return RingPos{pos % STAGES, static_cast<uint32_t>((pos / STAGES) & 1)};
}
template <int STAGES>
__device__ __forceinline__ RingPos ring_next(RingPos r) {
  if (++r.slot == STAGES) {
    r.slot = 0;
    r.phase ^= 1u;
  }
  return r;
}

// Masks the scores of keys outside [lo, hi] (tile-relative: element i is key k0 + i):
// one compare with a constant and one select per score without a window, an
// unsigned range check with a window.
__device__ __forceinline__ void apply_mask(float (&s)[BN], int hi, int lo, bool window) {
  if (window) {
    const uint32_t span = static_cast<uint32_t>(hi - lo);
#pragma unroll
    for (int i = 0; i < BN; ++i)
      if (static_cast<uint32_t>(i - lo) > span) s[i] = -CUDART_INF_F;
  } else {
#pragma unroll
    for (int i = 0; i < BN; ++i)
      if (i > hi) s[i] = -CUDART_INF_F;
  }
}

// Wait bounded by time only (used to drain work already in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kAttnWaitNs) break;
  }
}

// A work unit: 256 query rows (two Q tiles) of one (batch, head).
struct Unit {
  int q0, b, h, kvh;
  int Nq, Nk;              // this sequence's query / key counts
  int q_tok, k_tok;        // ragged batches: first token row of the sequence
  int jb0, je0, jb1, je1;  // key-tile range [jb, je) of Q tile 0 / 1 (empty: jb == je)
  int j_begin, j_end;      // the union, streamed through the K/V ring
};

__device__ __forceinline__ Unit make_unit(int w, const FwdParams& p, int n_qblk) {
  Unit u;
  int qblk, bh;
  if (p.causal) {  // longest q-blocks of every head first: causal work grows with q0
    const int rank = w / (p.B * p.Hq);
    bh = w % (p.B * p.Hq);
    qblk = n_qblk - 1 - rank;
  } else {         // q-blocks of one head are adjacent units and share its K/V in L2
    qblk = w % n_qblk;
    bh = w / n_qblk;
  }
  u.b = bh / p.Hq;
  u.h = bh % p.Hq;
  u.kvh = u.h / p.group;
  u.q0 = qblk * (BM * NQT);
  if (p.varlen) {
    const int qs = __ldg(p.cu_q + u.b), qe = __ldg(p.cu_q + u.b + 1);
    const int ks = __ldg(p.cu_k + u.b), ke = __ldg(p.cu_k + u.b + 1);
    u.q_tok = qs;
    u.k_tok = ks;
    u.Nq = qe - qs;
    u.Nk = ke - ks;
    // a slice outside the tensors, or longer than the unit list covers, is
    // dropped (nothing read or written for it) and reported
    if (qs < 0 || qe < qs || qe > p.total_q || ks < 0 || ke < ks || ke > p.total_k || u.Nq > p.Nq) {
      if (qblk == 0 && u.h == 0) atomicCAS(p.err, 0, ATTN_ERR_SEQLEN);
      u.Nq = 0;
      u.Nk = 0;
    }
  } else {
    u.q_tok = u.k_tok = 0;
    u.Nq = p.Nq;
    u.Nk = p.Nk;
  }
  const int off = u.Nk - u.Nq;  // bottom-right diagonal offset
  int jb[NQT], je[NQT];
#pragma unroll
  for (int t = 0; t < NQT; ++t) {
    jb[t] = je[t] = 0;
    const int r0 = u.q0 + t * BM;
    if (r0 >= u.Nq) continue;
    const int r1 = min(r0 + BM - 1, u.Nq - 1);
    int hi = u.Nk;
    if (p.causal) hi = min(hi, r1 + off + 1);
    int lo = 0;
    if (p.window > 0) lo = max(0, r0 + off - p.window + 1);
    if (hi > lo) {
      jb[t] = lo / BN;
      je[t] = (hi + BN - 1) / BN;
    }
  }
  u.jb0 = jb[0];
  u.je0 = je[0];
  u.jb1 = jb[1];
  u.je1 = je[1];
  u.j_begin = u.j_end = 0;
#pragma unroll
  for (int t = 0; t < NQT; ++t) {
    if (je[t] > jb[t]) {
      u.j_begin = (u.j_end > u.j_begin) ? min(u.j_begin, jb[t]) : jb[t];
      u.j_end = max(u.j_end, je[t]);
    }
  }
  return u;
}

// The unit a CTA takes in pass `pass` over the unit list: passes deal the units
// to the CTAs alternately from the first and from the last CTA, which evens out
// the work of longest-first (causal) lists.  Units grow with the pass, so a
// CTA is done at its first unit past the end.
__device__ __forceinline__ int unit_of_pass(int pass) {
  const int c = (pass & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  return pass * static_cast<int>(gridDim.x) + c;
}

__device__ __forceinline__ void own_range(const Unit& u, int t, int& jb, int& je) {
  jb = t == 0 ? u.jb0 : u.jb1;
  je = t == 0 ? u.je0 : u.je1;
}

template <int HD, bool F16, bool CAP, bool QK8>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<HD, F16, QK8>;
  constexpr int KBLKS = C::KBLKS;
  constexpr int TILE_BYTES = C::TILE_BYTES;
  constexpr int QK_SLABS = C::QK_SLABS;
  constexpr int QK_BOX = C::QK_BOX;
  constexpr int QK_TILE_BYTES = C::QK_TILE_BYTES;
  constexpr int STAGES = C::STAGES;
  constexpr int SMEM_Q = C::SMEM_Q;
  constexpr int SMEM_RING = C::SMEM_RING;
  constexpr int SMEM_BAR = C::SMEM_BAR;
  constexpr int SMEM_MISC = C::SMEM_MISC;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  const int warp = warp_id_uniform();
  const int lane = static_cast<int>(lane_id());

  // ---- barriers (phases run on across the units a CTA processes)
  constexpr int NQB = C::NQB;
  constexpr int B0 = 2 * NQB + 1;                       // first barrier after the Q and done barriers
  auto bar_q_full = [&](int qb) { return sb + SMEM_BAR + 8u * qb; };          // Q tile in buffer qb landed
  auto bar_q_empty = [&](int qb) { return sb + SMEM_BAR + 8u * (NQB + qb); }; // its last S done
  const uint32_t bar_mma_done = sb + SMEM_BAR + 8u * (2 * NQB);               // every MMA issued has completed
  auto bar_kv_full = [&](int s) { return sb + SMEM_BAR + 8u * (B0 + s); };
  auto bar_kv_empty = [&](int s) { return sb + SMEM_BAR + 8u * (B0 + STAGES + s); };
  auto bar_t = [&](int kind, int t) { return sb + SMEM_BAR + 8u * (B0 + 2 * STAGES + kind * NQT + t); };
  auto bar_s_full = [&](int t) { return bar_t(0, t); };   // S_t of a key tile in TMEM
  auto bar_p_lo = [&](int t) { return bar_t(1, t); };     // P_t keys 0-63 in TMEM (+ O_t rescaled)
  auto bar_p_hi = [&](int t) { return bar_t(2, t); };     // P_t keys 64-127 in TMEM
  auto bar_o_full = [&](int t) { return bar_t(3, t); };   // O_t of a unit complete
  auto bar_o_empty = [&](int t) { return bar_t(4, t); };  // epilogue has read O_t
  auto bar_stats_full = [&](int t) { return bar_t(5, t); };   // a unit's 1 / l of Q tile t in smem
  auto bar_stats_empty = [&](int t) { return bar_t(6, t); };  // the epilogue warps have read them
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_MISC + 4);
  volatile uint32_t* turn = reinterpret_cast<volatile uint32_t*>(smem + SMEM_MISC + 8);

  const int n_qblk = (p.Nq + BM * NQT - 1) / (BM * NQT);
  const int n_units = n_qblk * p.Hq * p.B;

  if (threadIdx.x == 0) {
    for (int qb = 0; qb < NQB; ++qb) {
      mbar_init(bar_q_full(qb), 1);
      mbar_init(bar_q_empty(qb), 1);   // released by the issuer of the tile it holds
    }
    mbar_init(bar_mma_done, NQT);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), NQT);   // released once both Q tiles are done with it
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(bar_s_full(t), 1);
      mbar_init(bar_p_lo(t), BM / 32);   // one arrival per softmax warp
      mbar_init(bar_p_hi(t), BM / 32);
      mbar_init(bar_o_full(t), 1);
      mbar_init(bar_o_empty(t), BM / 32);      // one arrival per epilogue warp
      mbar_init(bar_stats_full(t), BM / 32);   // one arrival per softmax warp
      mbar_init(bar_stats_empty(t), BM / 32);  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    *turn = 0;
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

  if (warp >= WARP_MMA) {
    setmaxnreg_dec<Regs<HD, CAP>::CTRL>();
    if (warp == WARP_TMA) {
      // ================================================================ producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        const uint64_t once_policy = l2_policy_evict_first();   // Q: read once
        const uint64_t keep_policy = l2_policy_evict_last();    // K/V: read by every q-block of a head
        int it = 0;   // ring position (runs on across units)
        int nql = 0;  // Q tiles loaded so far (tile t of the n-th unit with work is load 2n + t)
        bool ok = true;
        // Q tile t of the current unit into buffer nql % NQB, once the tile it held is done
        auto load_q = [&](const Unit& u, int t) -> bool {
          const int qb = nql % NQB, use = nql / NQB;
          if (use > 0 && !mbar_wait(bar_q_empty(qb), (use - 1) & 1, abort_flag, p.err)) return false;
          mbar_arrive_expect_tx(bar_q_full(qb), QK_TILE_BYTES);
          for (int kb = 0; kb < QK_SLABS; ++kb)
            if (p.varlen)
              tma_load_3d_hint(sb + SMEM_Q + qb * QK_TILE_BYTES + kb * KBLK_BYTES, &tm_q, bar_q_full(qb),
                               kb * QK_BOX, u.h, u.q_tok + u.q0 + t * BM, once_policy);
            else
              tma_load_3d_hint(sb + SMEM_Q + qb * QK_TILE_BYTES + kb * KBLK_BYTES, &tm_q, bar_q_full(qb),
                               kb * QK_BOX, u.q0 + t * BM, u.b * p.Hq + u.h, once_policy);
          ++nql;
          return true;
        };
        for (int pass = 0, w = unit_of_pass(0); w < n_units && ok; w = unit_of_pass(++pass)) {
          const Unit u = make_unit(w, p, n_qblk);
          if (u.j_end <= u.j_begin) continue;
          // Q tile 0 (its buffer freed a unit ago), the first K/V pair, then Q tile 1 (its
          // buffer is the previous unit's tile 0), so that tile 0 can start while tile 1 waits
          if (!load_q(u, 0)) { ok = false; break; }
          for (int j = u.j_begin; j < u.j_end && ok; ++j) {
            if (j == u.j_begin + 1 && !load_q(u, 1)) { ok = false; break; }
            for (int kv = 0; kv < 2; ++kv, ++it) {
              const int s = it % STAGES, use = it / STAGES;
              if (use > 0 && !mbar_wait(bar_kv_empty(s), (use - 1) & 1, abort_flag, p.err)) {
                ok = false;
                break;
              }
              // K: QK_SLABS slabs of QK_BOX elements (E4M3 K fills half a slot); V: KBLKS bf16 slabs
              const int slabs = kv ? KBLKS : QK_SLABS;
              const int box_x = kv ? 64 : QK_BOX;
              mbar_arrive_expect_tx(bar_kv_full(s), kv ? TILE_BYTES : QK_TILE_BYTES);
              const CUtensorMap* m = kv ? &tm_v : &tm_k;
              for (int kb = 0; kb < slabs; ++kb)
                if (p.varlen)
                  tma_load_3d_hint(sb + SMEM_RING + s * TILE_BYTES + kb * KBLK_BYTES, m, bar_kv_full(s),
                                   kb * box_x, u.kvh, u.k_tok + j * BN, keep_policy);
                else
                  tma_load_3d_hint(sb + SMEM_RING + s * TILE_BYTES + kb * KBLK_BYTES, m, bar_kv_full(s),
                                   kb * box_x, j * BN, u.b * p.Hkv + u.kvh, keep_policy);
            }
          }
          if (ok && u.j_end == u.j_begin + 1 && !load_q(u, 1)) { ok = false; break; }  // one-tile unit
        }
        if (!ok) {  // give up: let the copies already issued land before the CTA exits
          for (int i = max(0, nql - NQB); i < nql; ++i) drain_wait(bar_q_full(i % NQB), (i / NQB) & 1);
          for (int i = max(0, it - STAGES); i < it; ++i) drain_wait(bar_kv_full(i % STAGES), (i / STAGES) & 1);
        }
      }
    } else if (warp < WARP_MMA + NQT) {
      // ================================================================ MMA issuers
      // Warp WARP_MMA + t issues the MMAs of Q tile t; per key tile j its step is
      // PV_t(j) (P_t from tensor memory) then S_t(j+1).  The tensor core takes a
      // 128 x 128 x 16 MMA about every 64 cycles and holds the issuing thread for
      // most of that, so the two issuers take strict turns, step by step
      // (t = 0, 1, 0, 1, ...), and do everything but the MMAs outside their turn:
      // waits for ring slots, the epilogue and P's first half before it (its second
      // half inside), commits and slot releases after.  One issuer's bookkeeping then overlaps the
      // other's MMAs, and the tensor pipe sees the MMAs of one step together, so
      // S_t(j+1) is not held back behind the other tile's MMAs.  The turn order
      // only sets priority (the two Q tiles share no tensor memory and each issuer
      // releases ring slots for its own uses); the turn passes through a
      // shared-memory counter.  The whole warp runs the loop converged (its
      // descriptors and addresses warp-uniform); lane 0 issues.  MMAs of one
      // thread execute in issue order, which orders S_t(j+1) after PV_t(j)
      // (P_t aliases S_t).
      const int t = warp - WARP_MMA;
      {
        const uint32_t elect = lane == 0 ? 1u : 0u;  // the lane that issues
        auto wait_full = [&](RingPos r) { return mbar_wait(bar_kv_full(r.slot), r.phase, abort_flag, p.err); };
        // bounded spin until the turn counter reaches `seq`
        auto wait_turn = [&](uint32_t seq) {
          if (*turn == seq) return true;
          const unsigned long long t0 = global_ns();
          for (uint32_t it = 1;; ++it) {
            if (*turn == seq) return true;
            if ((it & 63u) == 0u) {
              if (*abort_flag) return false;
              if (global_ns() - t0 > kAttnWaitNs) {
                *abort_flag = 1;
                atomicCAS(p.err, 0, ATTN_ERR_TIMEOUT);
                return false;
              }
            }
          }
        };
        const uint64_t k_desc0 = smem_desc_sw128(sb + SMEM_RING, 16, 1024);
        const uint64_t v_desc0 = smem_desc_sw128(sb + SMEM_RING, KBLK_BYTES, 1024);
        auto k_desc = [&](RingPos r) { return desc_add(k_desc0, static_cast<uint32_t>(r.slot * TILE_BYTES) >> 4); };
        auto v_desc = [&](RingPos r) { return desc_add(v_desc0, static_cast<uint32_t>(r.slot * TILE_BYTES) >> 4); };
        int it_base = 0;                      // ring position of the current unit's first K tile
        int nq = 0;                           // units with work so far
        int n_own = 0;                        // own key tiles so far (phase of s_full / p_lo / p_hi)
        int n_out = 0;                        // units that produced O_t so far (phase of o_full / o_empty)
        uint32_t seq = static_cast<uint32_t>(t);  // this issuer's next turn
        bool ok = true;
        for (int pass = 0, w = unit_of_pass(0); w < n_units && ok; w = unit_of_pass(++pass)) {
          const Unit u = make_unit(w, p, n_qblk);
          if (u.j_end <= u.j_begin) continue;
          int jb, je;
          own_range(u, t, jb, je);
          if (je <= jb) jb = je = u.j_end;  // no own tiles: the slots are only released
          // this unit's Q tile t: load 2 nq + t
          const int qb = (2 * nq + t) % NQB;
          if (!mbar_wait(bar_q_full(qb), ((2 * nq + t) / NQB) & 1, abort_flag, p.err)) { ok = false; break; }
          const uint64_t q_desc = smem_desc_sw128(sb + SMEM_Q + qb * QK_TILE_BYTES, 16, 1024);
          if (jb < je) {  // first S of this unit (outside the turn order)
            const RingPos r = ring_pos<STAGES>(it_base + 2 * (jb - u.j_begin));
            if (!wait_full(r)) { ok = false; break; }
            tc_fence_after();
            issue_qk<HD, F16, QK8>(elect, tmem + s_col(t), q_desc, k_desc(r));
            mma_commit_if(elect, bar_s_full(t));
            mma_commit_if(elect, bar_kv_empty(r.slot));
            if (je - jb == 1) mma_commit_if(elect, bar_q_empty(qb));  // that was this unit's last S
          } else {
            mbar_arrive_if(elect, bar_q_empty(qb));
          }
          RingPos kj = ring_pos<STAGES>(it_base);  // K of key tile j
          for (int j = u.j_begin; j < u.j_end && ok; ++j) {
            const RingPos vj = ring_next<STAGES>(kj);  // V of key tile j
            const RingPos kn = ring_next<STAGES>(vj);  // K of key tile j + 1
            const bool own = j >= jb && j < je;
            const int lt = n_own + (j - jb);
            if (own) {
              // inputs of this step, before taking the turn: the ring slots (filled
              // long before in the steady state) first, P_t's first half last, so that
              // the turn follows the softmax's hand-over with as little delay as possible
              if (!wait_full(vj) || (j + 1 < je && !wait_full(kn))) { ok = false; break; }
              // PV overwrites O_t at the unit's first key tile: the epilogue of the
              // previous unit must have read it out.
              if (j == jb && n_out > 0 && !mbar_wait(bar_o_empty(t), (n_out - 1) & 1, abort_flag, p.err)) {
                ok = false;
                break;
              }
              if (!mbar_wait(bar_p_lo(t), lt & 1, abort_flag, p.err)) { ok = false; break; }
            }
            if (!wait_turn(seq)) { ok = false; break; }
            if (own) {
              tc_fence_after();
              issue_pv_half<HD, F16>(elect, tmem + o_col<HD>(t), tmem + s_col(t), v_desc(vj), j > jb, 0);
              if (!mbar_wait(bar_p_hi(t), lt & 1, abort_flag, p.err)) { ok = false; break; }
              tc_fence_after();
              issue_pv_half<HD, F16>(elect, tmem + o_col<HD>(t), tmem + s_col(t), v_desc(vj), true, BN / 32);
              if (j + 1 < je) issue_qk<HD, F16, QK8>(elect, tmem + s_col(t), q_desc, k_desc(kn));
            }
            *turn = seq + 1;  // the other issuer's turn
            seq += 2;
            if (own) {
              mma_commit_if(elect, bar_kv_empty(vj.slot));
              if (j + 1 == je) {
                mma_commit_if(elect, bar_o_full(t));
              } else {
                mma_commit_if(elect, bar_s_full(t));
                mma_commit_if(elect, bar_kv_empty(kn.slot));
                if (j + 2 == je) mma_commit_if(elect, bar_q_empty(qb));  // this unit's last S
              }
            } else {
              // outside this Q tile's range: release both slots once they are filled
              if (!wait_full(kj) || !wait_full(vj)) { ok = false; break; }
              mbar_arrive_if(elect, bar_kv_empty(kj.slot));
              mbar_arrive_if(elect, bar_kv_empty(vj.slot));
            }
            kj = kn;
          }
          if (je > jb) {
            n_own += je - jb;
            ++n_out;
          }
          it_base += 2 * (u.j_end - u.j_begin);
          ++nq;
        }
        // every MMA issued above must finish before tensor memory is released
        mma_commit_if(elect, bar_mma_done);
        drain_wait(bar_mma_done, 0);
      }
    }
  } else if (warp >= WARP_EPI) {
    setmaxnreg_dec<Regs<HD, CAP>::EPI>();
    // ================================================================ epilogue
    // Warp WARP_EPI + q takes rows [32q, 32q + 32) of each Q tile: once a unit's
    // last P V into O_t has completed it reads O_t out of tensor memory, hands
    // it back to the MMA issuer and writes O_t / l in the output type, while
    // the softmax warps already run the next unit.  Q tile 0, then Q tile 1, unit
    // by unit (the order in which they finish).
    const int quad = warp % 4;
    const uint32_t lane_sel = static_cast<uint32_t>(quad * 32) << 16;
    const float* stats = reinterpret_cast<const float*>(smem + C::SMEM_STATS);
    const uint64_t out_policy = l2_policy_evict_first();   // O is written once
    int n_unit = 0;          // units so far (phase of stats_full / stats_empty)
    int n_out[NQT] = {};     // units that produced O_t so far (phase of o_full / o_empty)
    bool ok = true;
    for (int pass = 0, w = unit_of_pass(0); w < n_units && ok; w = unit_of_pass(++pass)) {
      const Unit u = make_unit(w, p, n_qblk);
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        int jb, je;
        own_range(u, t, jb, je);
        ok = __all_sync(0xffffffffu, mbar_wait(bar_stats_full(t), n_unit & 1, abort_flag, p.err));
        if (!ok) break;
        const float inv_l = stats[t * BM + quad * 32 + lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_stats_empty(t));
        // the row's HD outputs, normalised and packed: word k holds outputs 2k, 2k + 1
        uint32_t wd[HD / 2];
        if (je > jb) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar_o_full(t), n_out[t] & 1, abort_flag, p.err));
          if (!ok) break;
          ++n_out[t];
          tc_fence_after();
          const uint32_t o_addr = tmem + lane_sel + o_col<HD>(t);
#pragma unroll
          for (int ch = 0; ch < HD / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(o_addr + ch * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k)
              wd[16 * ch + k] = pack2<F16>(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_o_empty(t));
        } else {
#pragma unroll
          for (int k = 0; k < HD / 2; ++k) wd[k] = 0u;   // no visible key: O = 0
        }
        const int row = u.q0 + t * BM + quad * 32 + lane;
        if (row < u.Nq) {
          const size_t orow_idx = p.varlen ? static_cast<size_t>(u.q_tok + row) * p.Hq + u.h
                                           : (static_cast<size_t>(u.b) * p.Hq + u.h) * p.Nq + row;
          uint16_t* orow = static_cast<uint16_t*>(p.o) + orow_idx * HD;
          if (p.o_align32) {
            // 32-byte stores: each thread writes its own row, so a warp's store touches 32
            // rows; whole 32-byte sectors halve the write requests of 16-byte stores
#pragma unroll
            for (int i = 0; i < HD / 16; ++i) st_global_v8_hint(orow + 16 * i, &wd[8 * i], out_policy);
          } else {
#pragma unroll
            for (int i = 0; i < HD / 8; ++i)
              reinterpret_cast<uint4*>(orow)[i] = make_uint4(wd[4 * i], wd[4 * i + 1], wd[4 * i + 2], wd[4 * i + 3]);
          }
        }
      }
      ++n_unit;
    }
  } else {
    setmaxnreg_inc<Regs<HD, CAP>::SOFTMAX>();
    // ================================================================ softmax
    const int t = (warp - WARP_SOFTMAX0) / 4;
    const int quad = warp % 4;
    const uint32_t lane_sel = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_sel + s_col(t);
    const uint32_t o_addr = tmem + lane_sel + o_col<HD>(t);
    const float c = p.scale_log2;
    int n_own = 0;  // own key tiles so far (phase of s_full)
    int n_unit = 0; // units so far (phase of stats_full / stats_empty)
    float* stats = reinterpret_cast<float*>(smem + C::SMEM_STATS);
    bool ok = true;
    for (int pass = 0, w = unit_of_pass(0); w < n_units && ok; w = unit_of_pass(++pass)) {
      const Unit u = make_unit(w, p, n_qblk);
      int jb, je;
      own_range(u, t, jb, je);
      const int n_tiles = max(0, je - jb);
      const int row = u.q0 + t * BM + quad * 32 + lane;
      const int off = u.Nk - u.Nq;
      // visible keys of this row: lo_r <= key <= hi_r
      const int diag = row + off;
      const int hi_r = p.causal ? min(diag, u.Nk - 1) : u.Nk - 1;
      const int lo_r = p.window > 0 ? diag - p.window + 1 : 0;
      // tile-uniform bounds: a K tile inside [tile_lo_max, tile_hi_min] needs no mask
      const int trow0 = u.q0 + t * BM;
      const int tile_hi_min = p.causal ? min(trow0 + off, u.Nk - 1) : u.Nk - 1;
      const int tile_lo_max = p.window > 0 ? trow0 + BM - 1 + off - p.window + 1 : 0;

      float m = -CUDART_INF_F;  // running max of scale*log2(e)*s (possibly stale)
      float l = 0.f;            // running sum of 2^(s*c - m)
      for (int jj = 0; jj < n_tiles; ++jj) {
        const int k0 = (jb + jj) * BN;
        const int lt = n_own + jj;
        ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full(t), lt & 1, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(s_addr + ch * 32, sr[ch]);
        tmem_wait_ld();
        float s[BN];
#pragma unroll
        for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(sr[i >> 5][i & 31]);
        const bool need_mask = k0 + BN - 1 > tile_hi_min || k0 < tile_lo_max;
        float mx[8];
        float rmax;   // the row maximum: of s * c (exp2 units), or of the capped scores
        if constexpr (CAP) {
          // Softcap: the warp caps this tile's scores with a polynomial when every raw
          // score of its 32 rows (masked ones included: they are finite here and are
          // set to -inf after the cap) lies in that polynomial's range.
          float mn[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            mx[g] = fmaxf(s[g], s[8 + g]);
            mn[g] = fminf(s[g], s[8 + g]);
          }
#pragma unroll
          for (int i = 16; i < BN; i += 16)
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              mx[g] = fmax3(mx[g], s[i + g], s[i + 8 + g]);
              mn[g] = fmin3(mn[g], s[i + g], s[i + 8 + g]);
            }
          const float rmax_raw = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
          const float rmin_raw = fmin3(fmin3(mn[0], mn[1], mn[2]), fmin3(mn[3], mn[4], mn[5]), fminf(mn[6], mn[7]));
          // the shortest polynomial every score of the warp's rows allows
          const bool fits_short =
              __all_sync(0xffffffffu, rmax_raw <= p.cap_smax_short && rmin_raw >= -p.cap_smax_short);
          const bool fits_long =
              __all_sync(0xffffffffu, rmax_raw <= p.cap_smax_long && rmin_raw >= -p.cap_smax_long);
          // s <- cap_post tanh(cap_pre s): the capped score in exp2 units, in place;
          // tanh is increasing, so rmax (the cap of the raw maximum) is the capped maximum
          rmax = rmax_raw;
          if (fits_short) {
            cap_polynomial<4>(s, &rmax, p.cap_short);
          } else if (fits_long) {
            cap_polynomial<6>(s, &rmax, p.cap_long);
          } else {     // through the exponential identity (two special-function operations)
#pragma unroll
            for (int i = 0; i < BN; ++i) s[i] = p.cap_post * tanh_exp(p.cap_pre * s[i]);
            rmax = p.cap_post * tanh_exp(p.cap_pre * rmax_raw);
          }
          if (need_mask) {
            apply_mask(s, hi_r - k0, lo_r - k0, p.window > 0);
#pragma unroll
            for (int g = 0; g < 8; ++g) mx[g] = fmaxf(s[g], s[8 + g]);
#pragma unroll
            for (int i = 16; i < BN; i += 16)
#pragma unroll
              for (int g = 0; g < 8; ++g) mx[g] = fmax3(mx[g], s[i + g], s[i + 8 + g]);
            rmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
          }
        } else {
          if (need_mask) {
            apply_mask(s, hi_r - k0, lo_r - k0, p.window > 0);
          }
#pragma unroll
          for (int g = 0; g < 8; ++g) mx[g] = fmaxf(s[g], s[8 + g]);
#pragma unroll
          for (int i = 16; i < BN; i += 16)
#pragma unroll
            for (int g = 0; g < 8; ++g) mx[g] = fmax3(mx[g], s[i + g], s[i + 8 + g]);
          rmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        }
        // the row maximum in exp2 units (the capped scores are in exp2 units already)
        const float cs = CAP ? 1.f : c;
        const float rmax_l2 = rmax * cs;
        const float m_new = fmaxf(m, rmax_l2);
        float alpha = 1.f;
        bool grow = false;
        if (jj == 0) {
          m = m_new;
        } else {
          grow = m_new > m + RESCALE_LOG2;
          if (grow) {
            alpha = ex2_approx(m - m_new);
            m = m_new;
          }
        }
        // O row *= alpha happens after P's first half is written (fewer live
        // registers) and before that half is handed over, so no PV of this tile
        // can start earlier.  PV of the previous tile is complete: its commit
        // preceded the S commit this thread waited on.
        const bool rescale = __any_sync(0xffffffffu, grow);
        l *= alpha;
        const float m_use = (m == -CUDART_INF_F) ? 0.f : m;
        // p = 2^(s cs - m), summed and packed to bf16 pairs; each half of the keys
        // is handed to the MMA issuer as soon as it is in tensor memory.
        const uint64_t c2 = f2_pack(cs, cs);
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // P columns [32*half, +32) = keys [64*half, +64)
#pragma unroll
          for (int qtr = 0; qtr < 2; ++qtr) {   // 16 columns = 32 keys at a time
            const int c0 = 64 * half + 32 * qtr;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(s[c0 + 2 * i], s[c0 + 2 * i + 1]), c2, nm2), x0, x1);
              const float p0 = ex2_approx(x0);
              const float p1 = ex2_approx(x1);
              sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
              pk[i] = pack2<F16>(p0, p1);
            }
            tmem_st16(s_addr + 32 * half + 16 * qtr, pk);
          }
          if (half == 0 && rescale) {
#pragma unroll 1
            for (int ch = 0; ch < HD / 32; ++ch) {
              uint32_t o[32];
              tmem_ld32(o_addr + ch * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(o_addr + ch * 32, o);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(half == 0 ? bar_p_lo(t) : bar_p_hi(t));
        }
        float sa, sb2, sc, sd;
        f2_unpack(sum2[0], sa, sb2);
        f2_unpack(sum2[1], sc, sd);
        l += (sa + sb2) + (sc + sd);
      }
      if (!ok) break;
      n_own += n_tiles;

      // ---- the row's normaliser 1 / l, handed to the epilogue warps, and LSE; a
      // sink adds 2^(sink - m) to the row sum (in the common maximum M = max(m,
      // sink)); a row with no visible key has O = 0 and LSE = sink
      float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      float lse_val = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      if (p.sinks != nullptr) {
        const float sink = __ldg(p.sinks + u.h);
        if (l > 0.f) {
          const float M = fmaxf(m, sink * 1.4426950408889634f);
          const float w = ex2_approx(m - M);
          const float lt = fmaf(l, w, ex2_approx(sink * 1.4426950408889634f - M));
          inv_l = w / lt;
          lse_val = (M + log2f(lt)) * 0.69314718055994531f;
        } else {
          inv_l = 0.f;
          lse_val = sink;
        }
      }
      inv_l *= p.o_scale;
      // the epilogue warps must have taken the previous unit's normalisers
      if (n_unit > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_stats_empty(t), (n_unit - 1) & 1, abort_flag, p.err));
        if (!ok) break;
      }
      stats[t * BM + quad * 32 + lane] = inv_l;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_stats_full(t));
      ++n_unit;
      if (row < u.Nq && p.lse != nullptr) {
        const size_t li = p.varlen ? static_cast<size_t>(u.h) * p.total_q + u.q_tok + row
                                   : (static_cast<size_t>(u.b) * p.Hq + u.h) * p.Nq + row;
        p.lse[li] = lse_val;
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

}  // namespace fwd_bf16

// --------------------------------------------------------------------- host
namespace fwd_bf16 {

template <int HD, bool F16, bool CAP, bool QK8 = false>
int launch_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                int Hkv, int Nq, int Nk, float scale, int causal, int window, int num_sms,
                cudaStream_t stream, int* err, const int* cu_q, const int* cu_k, int total_q,
                int total_k, float softcap, const float* sinks, float o_scale = 1.f) {
  using C = Cfg<HD, F16, QK8>;
  const CUtensorMapDataType dt = F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // Q and K: 16-bit, or E4M3 codes (one byte, 128 per 128-byte box row)
  const CUtensorMapDataType dt_qk = QK8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : dt;
  const uint32_t es_qk = QK8 ? 1u : 2u;
  CUtensorMap tq, tk, tv;
  const bool varlen = cu_q != nullptr;
  if (varlen) {  // packed [total, H, D]: 128 token rows of one head per box
    const uint32_t box[3] = {64, 1, 128};
    const uint32_t box_qk[3] = {static_cast<uint32_t>(C::QK_BOX), 1, 128};
    if (!encode_tiled_3d(&tq, dt_qk, q, HD, Hq, total_q, es_qk, box_qk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_3d(&tk, dt_qk, k, HD, Hkv, total_k, es_qk, box_qk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_3d(&tv, dt, v, HD, Hkv, total_k, 2, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  } else {       // [B*H, N, D]: 128 rows of one (batch, head) per box
    const uint32_t box[3] = {64, 128, 1};
    const uint32_t box_qk[3] = {static_cast<uint32_t>(C::QK_BOX), 128, 1};
    if (!encode_tiled_3d(&tq, dt_qk, q, HD, Nq, static_cast<uint64_t>(B) * Hq, es_qk, box_qk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_3d(&tk, dt_qk, k, HD, Nk, static_cast<uint64_t>(B) * Hkv, es_qk, box_qk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_3d(&tv, dt, v, HD, Nk, static_cast<uint64_t>(B) * Hkv, 2, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  static KernelSetup setup;
  if (const int rc = prepare_kernel(setup, attn_fwd_bf16_kernel<HD, F16, CAP, QK8>, C::SMEM_ALLOC); rc != ATTN_OK)
    return rc;
  // The warpgroups' setmaxnreg shares add up to 65536 registers, which the block's pool
  // (its registers per thread at launch x NTHREADS) must hold, or an `inc` never returns.
  static std::atomic<int> regs_ok{-1};
  if (regs_ok.load() < 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, attn_fwd_bf16_kernel<HD, F16, CAP, QK8>) != cudaSuccess) return ATTN_ERR_CUDA;
    regs_ok.store(fa.numRegs * NTHREADS >= 65536 ? 1 : 0);
  }
  if (regs_ok.load() != 1) return ATTN_ERR_CUDA;
  FwdParams prm;
  prm.o = o;
  prm.lse = lse;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.group = Hq / Hkv;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.causal = causal ? 1 : 0;
  prm.window = window > 0 ? window : 0;
  prm.err = err;
  prm.varlen = varlen ? 1 : 0;
  prm.cu_q = cu_q;
  prm.cu_k = cu_k;
  prm.total_q = total_q;
  prm.total_k = total_k;
  prm.cap_pre = CAP ? scale / softcap : 0.f;
  prm.cap_post = CAP ? softcap * 1.4426950408889634f : 0.f;
  // Softcap fast paths: cap_post tanh(a s) = s * sum_k (scale log2(e) t_k a^(2k)) (s^2)^k with
  // a = scale / softcap, valid while |a s| <= the fit's y_max.  A fit whose prescaled
  // coefficients are not all normal floats (an extreme scale / softcap ratio) stays disabled.
  auto prescale = [&](const double* t, int terms, double ymax, float* out, float* smax_out) {
    *smax_out = -1.f;
    for (int i = 0; i < terms; ++i) out[i] = 0.f;
    if (!CAP) return;
    const double a = static_cast<double>(scale) / softcap;
    const double c2 = static_cast<double>(scale) * 1.4426950408889634;
    bool ok = true;
    double ak = 1.0;
    for (int i = 0; i < terms; ++i) {
      const double u = c2 * t[i] * ak;
      ok = ok && std::isfinite(u) && std::fabs(u) >= 1e-36 && std::fabs(u) <= 1e36;  // normal floats
      out[i] = static_cast<float>(u);
      ak *= a * a;
    }
    const double smax = ymax / a;
    if (ok && std::isfinite(smax) && smax < 1e15) *smax_out = static_cast<float>(smax);
  };
  prescale(kTanhPolyShort, 4, kTanhPolyShortYMax, prm.cap_short, &prm.cap_smax_short);
  prescale(kTanhPolyLong, 6, kTanhPolyLongYMax, prm.cap_long, &prm.cap_smax_long);
  prm.sinks = sinks;
  prm.o_scale = o_scale;
  prm.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
  // persistent: at most one CTA per SM, each walking units blockIdx.x, +gridDim.x, ...
  const long long n_qblk = (Nq + BM * NQT - 1) / (BM * NQT);
  const long long units = n_qblk * Hq * B;
  if (units > 0x7fffffffLL) return ATTN_ERR_DIM;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  attn_fwd_bf16_kernel<HD, F16, CAP, QK8><<<grid, NTHREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, prm);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace fwd_bf16

int launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, int f16, float scale, int causal, int window,
                  int num_sms, cudaStream_t stream, int* err, const int* cu_q, const int* cu_k,
                  int total_q, int total_k, float softcap, const float* sinks) {
  using fwd_bf16::launch_impl;
#define ATTN_TC_ARGS q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, num_sms, stream, err, \
                     cu_q, cu_k, total_q, total_k, softcap, sinks
  const bool cap = softcap > 0.f;
  if (cap && f16) return ATTN_ERR_HEAD_DIM;  // the softcap instances are bf16 only
  if (D == 64 && !f16) return cap ? launch_impl<64, false, true>(ATTN_TC_ARGS) : launch_impl<64, false, false>(ATTN_TC_ARGS);
  if (D == 128 && !f16) return cap ? launch_impl<128, false, true>(ATTN_TC_ARGS) : launch_impl<128, false, false>(ATTN_TC_ARGS);
  if (D == 64 && f16) return launch_impl<64, true, false>(ATTN_TC_ARGS);
  if (D == 128 && f16) return launch_impl<128, true, false>(ATTN_TC_ARGS);
#undef ATTN_TC_ARGS
  return ATTN_ERR_HEAD_DIM;
}

// ---------------------------------------------------------------- fp8 prefill
namespace fwd_bf16 {

// E4M3 codes -> bf16 values, 16 codes per thread and step (one 16-byte load, two
// 16-byte stores).  Exact: every E4M3 value (NaN included) is a bf16 value, and
// the conversion goes through f16, which also holds every E4M3 value exactly.
__global__ void __launch_bounds__(256) e4m3_to_bf16_kernel(const uint4* __restrict__ in,
                                                           uint4* __restrict__ out, size_t n16) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 c = __ldcs(in + i);  // read once
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t r[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // two codes (bytes 2*half, 2*half + 1 of w[k]) -> f16x2 -> two floats -> bf16x2
        const uint16_t pair = static_cast<uint16_t>(w[k] >> (16 * half));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        float lo, hi;
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
            : "=f"(lo), "=f"(hi) : "r"(h2));
        r[2 * k + half] = pack_bf16x2(lo, hi);
      }
    }
    out[2 * i] = make_uint4(r[0], r[1], r[2], r[3]);
    out[2 * i + 1] = make_uint4(r[4], r[5], r[6], r[7]);
  }
}

}  // namespace fwd_bf16

size_t fwd_fp8_workspace_bytes(int B, int Hkv, int Nk, int D) {
  return static_cast<size_t>(B) * Hkv * Nk * D * 2;
}

int launch_fwd_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                   float v_scale, void* o, float* lse, void* workspace, int B, int Hq, int Hkv,
                   int Nq, int Nk, int D, float scale, int causal, int window, int num_sms,
                   cudaStream_t stream, int* err) {
  if (D != 128) return ATTN_ERR_HEAD_DIM;
  // V widened to bf16 in the workspace, then the forward with S on E4M3 Q/K; the
  // Q and K scales fold into the score scale, the V scale into the normaliser.
  const size_t n16 = static_cast<size_t>(B) * Hkv * Nk * D / 16;
  const long long want = static_cast<long long>((n16 + 255) / 256);
  const int grid = static_cast<int>(want < 4LL * num_sms ? (want > 0 ? want : 1) : 4LL * num_sms);
  fwd_bf16::e4m3_to_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(v),
                                                         static_cast<uint4*>(workspace), n16);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  return fwd_bf16::launch_impl<128, false, false, true>(q, k, workspace, o, lse, B, Hq, Hkv, Nq, Nk,
                                                       scale * q_scale * k_scale, causal, window,
                                                       num_sms, stream, err, nullptr, nullptr, 0, 0,
                                                       0.f, nullptr, v_scale);
}

}  // namespace attn

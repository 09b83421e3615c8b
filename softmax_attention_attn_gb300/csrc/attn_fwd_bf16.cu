// attn_fwd_bf16.cu — bf16 fused attention forward for sm_103a on tcgen05.
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
//   * one CTA owns two 128-row Q tiles of one (batch, head) and streams 128-key
//     K/V tiles through a 4-slot TMA ring (128-byte swizzle, mbarrier
//     transaction counts);
//   * warp 9 (one elected thread) issues tcgen05.mma: S_t = Q_t K^T into tensor
//     memory (fp32, 128 columns per Q tile), then O_t += P_t V with P read from
//     tensor memory (the TS form) and V from shared memory (MN-major operand);
//   * warps 0-3 and 4-7 are the softmax warpgroups of Q tile 0 and 1: thread r
//     owns row r, loads its 128 scores from tensor memory, applies the mask,
//     updates the running max / sum in the exp2 domain, rescales its O row in
//     tensor memory when the max grew by more than 2^8 (otherwise the stale max
//     is kept; the final normalisation is exact either way), writes P as bf16
//     over its S columns and signals the MMA warp;
//   * warp 8 (one elected thread) is the TMA producer;
//   * the epilogue (same softmax threads) divides by the row sum, rounds O to
//     bf16 and writes O and LSE.
//
// The two Q tiles ping-pong: while warpgroup 0 runs the softmax of tile j the
// tensor core computes PV_1(j-1) and S_1(j), and vice versa.
//
// Tensor memory (512 columns): S_0 [0,128) S_1 [128,256) O_0 [256,384) O_1 [384,512);
// P_t aliases the first 64 columns of S_t (two bf16 per 32-bit column).
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace fwd_bf16 {

constexpr int BM = 128;                      // query rows per Q tile
constexpr int BN = 128;                      // keys per K/V tile
constexpr int HD = 128;                      // head dimension
constexpr int NQT = 2;                       // Q tiles per CTA
constexpr int STAGES = 4;                    // K/V ring slots (one K or one V tile each)
constexpr int KBLK_BYTES = BN * 64 * 2;      // 64-column (128-byte) slab of a 128-row tile
constexpr int TILE_BYTES = 2 * KBLK_BYTES;   // 128 x 128 bf16
constexpr int SMEM_Q = 0;
constexpr int SMEM_RING = SMEM_Q + NQT * TILE_BYTES;
constexpr int SMEM_BAR = SMEM_RING + STAGES * TILE_BYTES;
constexpr int NUM_BARS = 2 + 2 * STAGES + 4 * NQT;
constexpr int SMEM_MISC = SMEM_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = SMEM_MISC + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
constexpr int NUM_SOFTMAX_WARPS = 4 * NQT;
constexpr int WARP_TMA = NUM_SOFTMAX_WARPS;
constexpr int WARP_MMA = NUM_SOFTMAX_WARPS + 1;
constexpr int NTHREADS = (NUM_SOFTMAX_WARPS + 2) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;         // keep a stale max while the growth is <= 2^8
constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, BN, 0);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, HD, 1);

static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ uint32_t s_col(int t) { return static_cast<uint32_t>(t * BN); }
__device__ __forceinline__ uint32_t o_col(int t) { return static_cast<uint32_t>(NQT * BN + t * HD); }

// S (tmem) = Q_tile (smem) x K_tile^T (smem); both K-major, 128-byte swizzle.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t koff = static_cast<uint32_t>((kk >> 2) * KBLK_BYTES + (kk & 3) * 32);
    const uint64_t a = smem_desc_sw128(q_smem + koff, 16, 1024);
    const uint64_t b = smem_desc_sw128(k_smem + koff, 16, 1024);
    mma_bf16_ss(d_tmem, a, b, IDESC_QK, kk > 0 ? 1u : 0u);
  }
}

// O (tmem) (+)= P (tmem, bf16) x V_tile (smem, MN-major: d contiguous), for the
// 16-key steps kk in [kk0, kk0 + 4): one half of the tile's keys.
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                              bool accumulate, int kk0) {
#pragma unroll
  for (int kk = kk0; kk < kk0 + BN / 32; ++kk) {
    const uint64_t b = smem_desc_sw128(v_smem + static_cast<uint32_t>(kk * 16 * 128),
                                       KBLK_BYTES, 1024);
    mma_bf16_ts(d_tmem, p_tmem + static_cast<uint32_t>(kk * 8), b, IDESC_PV,
                (accumulate || kk > 0) ? 1u : 0u);
  }
}

// Wait bounded by time only (used to drain work already in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kAttnWaitNs) break;
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  const int warp = warp_id_uniform();
  const int lane = static_cast<int>(lane_id());

  const uint32_t bar_q = sb + SMEM_BAR;
  const uint32_t bar_mma_done = sb + SMEM_BAR + 8;
  auto bar_kv_full = [&](int s) { return sb + SMEM_BAR + 8u * (2 + s); };
  auto bar_kv_empty = [&](int s) { return sb + SMEM_BAR + 8u * (2 + STAGES + s); };
  auto bar_s_full = [&](int t) { return sb + SMEM_BAR + 8u * (2 + 2 * STAGES + t); };
  // P of Q tile t is handed over in two halves (keys 0-63, keys 64-127)
  auto bar_p_lo = [&](int t) { return sb + SMEM_BAR + 8u * (2 + 2 * STAGES + NQT + t); };
  auto bar_p_hi = [&](int t) { return sb + SMEM_BAR + 8u * (2 + 2 * STAGES + 2 * NQT + t); };
  auto bar_o_full = [&](int t) { return sb + SMEM_BAR + 8u * (2 + 2 * STAGES + 3 * NQT + t); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_MISC + 4);

  // ---- work unit: (batch b, head h, 256 query rows starting at q0)
  const int qblk = p.causal ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  const int h = static_cast<int>(blockIdx.y);
  const int b = static_cast<int>(blockIdx.z);
  const int kvh = h / p.group;
  const int q0 = qblk * (BM * NQT);
  const int off = p.Nk - p.Nq;  // bottom-right diagonal offset
  int kv_hi = p.Nk;             // exclusive key bound of the CTA
  if (p.causal) kv_hi = min(kv_hi, min(q0 + BM * NQT - 1, p.Nq - 1) + off + 1);
  int kv_lo = 0;
  if (p.window > 0) kv_lo = max(0, q0 + off - p.window + 1);
  int j_begin = 0, n_tiles = 0;
  if (kv_hi > kv_lo) {
    j_begin = kv_lo / BN;
    n_tiles = (kv_hi + BN - 1) / BN - j_begin;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_mma_done, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(bar_s_full(t), 1);
      mbar_init(bar_p_lo(t), BM / 32);   // one arrival per softmax warp
      mbar_init(bar_p_hi(t), BM / 32);
      mbar_init(bar_o_full(t), 1);
    }
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

  if (warp == WARP_TMA) {
    // ================================================================ producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar_q, NQT * TILE_BYTES);
      for (int t = 0; t < NQT; ++t)
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(sb + SMEM_Q + t * TILE_BYTES + kb * KBLK_BYTES, &tm_q, bar_q, kb * 64,
                      q0 + t * BM, b * p.Hq + h);
      int it = 0;
      bool ok = true;
      for (int jj = 0; jj < n_tiles && ok; ++jj) {
        const int krow = (j_begin + jj) * BN;
        for (int kv = 0; kv < 2; ++kv, ++it) {
          const int s = it % STAGES, u = it / STAGES;
          if (u > 0 && !mbar_wait(bar_kv_empty(s), (u - 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_kv_full(s), TILE_BYTES);
          const CUtensorMap* m = kv ? &tm_v : &tm_k;
          for (int kb = 0; kb < 2; ++kb)
            tma_load_3d(sb + SMEM_RING + s * TILE_BYTES + kb * KBLK_BYTES, m, bar_kv_full(s),
                        kb * 64, krow, b * p.Hkv + kvh);
        }
      }
      if (!ok) {  // give up: let the copies already issued land before the CTA exits
        drain_wait(bar_q, 0);
        for (int i = max(0, it - STAGES); i < it; ++i) drain_wait(bar_kv_full(i % STAGES), (i / STAGES) & 1);
      }
    }
  } else if (warp == WARP_MMA) {
    // ================================================================ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait(bar_q, 0, abort_flag, p.err);
      int it = 0;
      if (ok) ok = mbar_wait(bar_kv_full(0), 0, abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < NQT; ++t) {
          issue_qk(tmem + s_col(t), sb + SMEM_Q + t * TILE_BYTES, sb + SMEM_RING);
          mma_commit(bar_s_full(t));
        }
        mma_commit(bar_kv_empty(0));
      }
      it = 1;
      for (int jj = 0; jj < n_tiles && ok; ++jj) {
        const int vs = it % STAGES, vu = it / STAGES;
        ++it;
        const bool last = (jj == n_tiles - 1);
        int ks = 0, ku = 0;
        if (!last) {
          ks = it % STAGES;
          ku = it / STAGES;
          ++it;
        }
        if (!mbar_wait(bar_kv_full(vs), vu & 1, abort_flag, p.err)) { ok = false; break; }
        for (int t = 0; t < NQT; ++t) {
          const uint32_t vsm = sb + SMEM_RING + vs * TILE_BYTES;
          if (!mbar_wait(bar_p_lo(t), jj & 1, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          issue_pv_half(tmem + o_col(t), tmem + s_col(t), vsm, jj > 0, 0);
          if (!mbar_wait(bar_p_hi(t), jj & 1, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          issue_pv_half(tmem + o_col(t), tmem + s_col(t), vsm, true, BN / 32);
          if (t == NQT - 1) mma_commit(bar_kv_empty(vs));
          if (last) {
            mma_commit(bar_o_full(t));
          } else {
            if (t == 0) {
              if (!mbar_wait(bar_kv_full(ks), ku & 1, abort_flag, p.err)) { ok = false; break; }
              tc_fence_after();
            }
            issue_qk(tmem + s_col(t), sb + SMEM_Q + t * TILE_BYTES, sb + SMEM_RING + ks * TILE_BYTES);
            mma_commit(bar_s_full(t));
            if (t == NQT - 1) mma_commit(bar_kv_empty(ks));
          }
        }
      }
      // every MMA issued above must finish before tensor memory is released
      mma_commit(bar_mma_done);
      drain_wait(bar_mma_done, 0);
    }
  } else {
    // ================================================================ softmax + epilogue
    const int t = warp / 4;
    const int quad = warp % 4;
    const int row = q0 + t * BM + quad * 32 + lane;
    const uint32_t lane_sel = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_sel + s_col(t);
    const uint32_t o_addr = tmem + lane_sel + o_col(t);
    const float c = p.scale_log2;

    // visible keys of this row: lo_r <= key <= hi_r
    const int diag = row + off;
    const int hi_r = p.causal ? min(diag, p.Nk - 1) : p.Nk - 1;
    const int lo_r = p.window > 0 ? diag - p.window + 1 : 0;
    // tile-uniform bounds: a K tile inside [tile_lo_max, tile_hi_min] needs no mask
    const int trow0 = q0 + t * BM;
    const int tile_hi_min = p.causal ? min(trow0 + off, p.Nk - 1) : p.Nk - 1;
    const int tile_lo_max = p.window > 0 ? trow0 + BM - 1 + off - p.window + 1 : 0;

    float m = -CUDART_INF_F;  // running max of scale*log2(e)*s (possibly stale)
    float l = 0.f;            // running sum of 2^(s*c - m)
    bool ok = true;
    for (int jj = 0; jj < n_tiles; ++jj) {
      const int k0 = (j_begin + jj) * BN;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full(t), jj & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld32(s_addr + ch * 32, sr[ch]);
      tmem_wait_ld();
      float s[BN];
#pragma unroll
      for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(sr[i >> 5][i & 31]);
      if (k0 + BN - 1 > tile_hi_min || k0 < tile_lo_max) {
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const int key = k0 + i;
          if (key > hi_r || key < lo_r) s[i] = -CUDART_INF_F;
        }
      }
      float mx[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) mx[g] = fmaxf(s[g], s[8 + g]);
#pragma unroll
      for (int i = 16; i < BN; i += 16)
#pragma unroll
        for (int g = 0; g < 8; ++g) mx[g] = fmax3(mx[g], s[i + g], s[i + 8 + g]);
      const float rmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      const float m_new = fmaxf(m, rmax * c);
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
      // p = 2^(s*c - m), summed and packed to bf16 pairs; each half of the keys is
      // handed to the MMA warp as soon as it is in tensor memory.
      const uint64_t c2 = f2_pack(c, c);
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
            const uint64_t x2 = f2_fma(f2_pack(s[c0 + 2 * i], s[c0 + 2 * i + 1]), c2, nm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(s_addr + 32 * half + 16 * qtr, pk);
        }
        if (half == 0 && rescale) {
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
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

    // ---- epilogue: O / l -> bf16, LSE
    bool have_o = n_tiles > 0 && ok;
    if (have_o) {
      have_o = __all_sync(0xffffffffu, mbar_wait(bar_o_full(t), 0, abort_flag, p.err));
      if (have_o) tc_fence_after();
    }
    const bool row_ok = row < p.Nq;
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    __nv_bfloat16* orow = p.o + ((static_cast<size_t>(b) * p.Hq + h) * p.Nq + (row_ok ? row : 0)) * HD;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(o_addr + ch * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
    }
    if (row_ok && p.lse != nullptr) {
      const float lse = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Nq + row] = lse;
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
int launch_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int Hq, int Hkv, int Nq, int Nk, float scale, int causal, int window,
                    cudaStream_t stream, int* err) {
  using namespace fwd_bf16;
  CUtensorMap tq, tk, tv;
  const uint32_t box[3] = {64, 128, 1};
  if (!encode_tiled_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, HD, Nq, static_cast<uint64_t>(B) * Hq,
                       2, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k, HD, Nk, static_cast<uint64_t>(B) * Hkv,
                       2, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, HD, Nk, static_cast<uint64_t>(B) * Hkv,
                       2, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return ATTN_ERR_CUDA;
  static int attr_set_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_dev != dev) {
    if (cudaFuncSetAttribute(attn_fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_ALLOC) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_set_dev = dev;
  }
  FwdParams prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
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
  const dim3 grid((Nq + BM * NQT - 1) / (BM * NQT), Hq, B);
  attn_fwd_bf16_kernel<<<grid, NTHREADS, SMEM_ALLOC, stream>>>(tq, tk, tv, prm);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

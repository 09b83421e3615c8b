// attn_fwd_fp32.cu — fp32 fused attention forward on the FP32 SIMT pipes.
//
// Follows "Agent 帮我写 CUDA：一个 Softmax Attention 算子的开发全记录": the tiled
// kernel of section 四 (a block owns a tile of query rows, loops over K/V tiles
// held in shared memory and merges the online-softmax state across tiles), the
// 16-byte vector loads of section 五, and the head-dimension-specific
// compilation of section 六 (one instantiation per D).  Differences for sm_103a:
//   * each thread computes a 4x4 block of scores and a 4 x D/16 block of O
//     (register tiling instead of one warp per row); the softmax statistics are
//     reduced with half-warp shuffles;
//   * two CTAs share an SM (16 warps), so each keeps its shared memory to 112 KB
//     at D = 128: one K and one V buffer, filled by cp.async one phase ahead
//     (K of the next tile streams in during the softmax and P V of this tile, V
//     of the next tile during the next Q K^T), no padding.  Instead of the padded
//     rows of section 五, the 16-byte chunks of each K row are XOR-swizzled by the
//     row index, so the 16 K rows that a half-warp reads at one column fall into
//     different banks; Q, V and P reads are broadcasts or contiguous;
//   * exponentials use the exp2 form 2^(s*scale*log2 e - m);
//   * the Q K^T and P V products run as packed pairs (fma.rn.f32x2: two IEEE fp32
//     FMAs per instruction, so the FMA pipe is kept busy with half the issue slots
//     and the shared-memory loads issue in between).
// No TF32 or other reduced-precision arithmetic is used.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace fwd_fp32 {

constexpr int BM = 64;   // query rows per CTA
constexpr int BN = 64;   // keys per tile
constexpr int NT = 256;  // threads: 16 row groups x 16 column groups

template <int D>
struct Smem {
  static constexpr int Q = 0;                    // [BM][D]
  static constexpr int K = Q + BM * D;           // [BN][D], 16-byte chunks swizzled
  static constexpr int V = K + BN * D;           // [BN][D]
  static constexpr int P = V + BN * D;           // [BM][BN]
  static constexpr int FLOATS = P + BM * BN;
  static constexpr int BYTES = FLOATS * 4;
  static constexpr int CHUNKS = D / 4;           // 16-byte chunks per row
  static constexpr int SWZ = CHUNKS < 16 ? CHUNKS - 1 : 15;
};

// Float offset of the 16-byte chunk `c` of K row `r` (swizzled by the row).
template <int D>
__device__ __forceinline__ int k_off(int r, int c) {
  return r * D + ((c ^ (r & Smem<D>::SWZ)) << 2);
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  const uint32_t d = smem_u32(dst);
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// rows [row0, row0+64) of a [N, D] head into shared memory ([64][D]; K rows swizzled)
template <int D, bool SWIZZLE>
__device__ __forceinline__ void load_rows(float* dst, const float* head, int row0, int N) {
  constexpr int VEC = D / 4;  // float4 per row
  for (int i = threadIdx.x; i < 64 * VEC; i += NT) {
    const int r = i / VEC, c = i % VEC;
    const int gr = row0 + r;
    const bool valid = gr < N;
    float* d = SWIZZLE ? dst + k_off<D>(r, c) : dst + r * D + c * 4;
    cp_async16(d, head + static_cast<size_t>(valid ? gr : 0) * D + c * 4, valid);
  }
}

template <int D>
__global__ void __launch_bounds__(NT, 2) attn_fwd_fp32_kernel(const float* __restrict__ Q,
                                                             const float* __restrict__ K,
                                                             const float* __restrict__ V,
                                                             float* __restrict__ O,
                                                             float* __restrict__ LSE, int Hq, int Hkv,
                                                             int Nq, int Nk, float c, int causal,
                                                             int window) {
  using S = Smem<D>;
  constexpr int DC = D / 16;  // output columns per thread
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float* Qs = sm + S::Q;
  float* Ks = sm + S::K;
  float* Vs = sm + S::V;
  float* Ps = sm + S::P;

  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int qblk = causal ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / (Hq / Hkv);
  const int q0 = qblk * BM;
  const int off = Nk - Nq;
  const float* Qh = Q + (static_cast<size_t>(b) * Hq + h) * Nq * D;
  const float* Kh = K + (static_cast<size_t>(b) * Hkv + kvh) * Nk * D;
  const float* Vh = V + (static_cast<size_t>(b) * Hkv + kvh) * Nk * D;

  int kv_hi = Nk;
  if (causal) kv_hi = min(kv_hi, min(q0 + BM - 1, Nq - 1) + off + 1);
  int kv_lo = 0;
  if (window > 0) kv_lo = max(0, q0 + off - window + 1);
  int j_begin = 0, n_tiles = 0;
  if (kv_hi > kv_lo) {
    j_begin = kv_lo / BN;
    n_tiles = (kv_hi + BN - 1) / BN - j_begin;
  }
  const int tile_hi_min = causal ? min(q0 + off, Nk - 1) : Nk - 1;
  const int tile_lo_max = window > 0 ? q0 + BM - 1 + off - window + 1 : 0;

  // cp.async groups in issue order: {Q, K_0}, {V_0}, then per tile j: {K_j+1} after
  // Q K^T_j and {V_j+1} after P V_j.  Waiting for all but the newest group therefore
  // always completes the buffer about to be read.
  if (n_tiles > 0) {
    load_rows<D, false>(Qs, Qh, q0, Nq);
    load_rows<D, true>(Ks, Kh, j_begin * BN, Nk);
  }
  cp_async_commit();
  if (n_tiles > 0) load_rows<D, false>(Vs, Vh, j_begin * BN, Nk);
  cp_async_commit();

  // O accumulators as packed pairs of adjacent output columns (fma.rn.f32x2)
  constexpr int DP = DC / 2;
  float m[4], l[4];
  uint64_t acc[4][DP];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -CUDART_INF_F;
    l[i] = 0.f;
#pragma unroll
    for (int d = 0; d < DP; ++d) acc[i][d] = 0ull;
  }

  for (int jj = 0; jj < n_tiles; ++jj) {
    cp_async_wait<1>();
    __syncthreads();  // K_j (and Q) visible; everyone is done with P V_j-1 (P buffer free)

    // ---- scores: rows ty*4+i, keys tx+16*n.  Packed fp32 pairs (fma.rn.f32x2, two
    // IEEE fp32 FMAs per instruction): s2 holds the partial sums over even and odd d,
    // added at the end; a 16-byte load gives the pairs (d, d+1) and (d+2, d+3).
    uint64_t s2[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int n = 0; n < 4; ++n) s2[i][n] = 0ull;
#pragma unroll 4
    for (int d = 0; d < D; d += 4) {
      ulonglong2 qv[4], kv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[i] = *reinterpret_cast<const ulonglong2*>(Qs + (ty * 4 + i) * D + d);
#pragma unroll
      for (int n = 0; n < 4; ++n) kv[n] = *reinterpret_cast<const ulonglong2*>(Ks + k_off<D>(tx + 16 * n, d >> 2));
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          s2[i][n] = f2_fma(qv[i].x, kv[n].x, s2[i][n]);
          s2[i][n] = f2_fma(qv[i].y, kv[n].y, s2[i][n]);
        }
    }
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        float e, o;
        f2_unpack(s2[i][n], e, o);
        s[i][n] = e + o;
      }
    __syncthreads();  // everyone is done with K_j: stream K_j+1 in during the softmax and P V
    if (jj + 1 < n_tiles) load_rows<D, true>(Ks, Kh, (j_begin + jj + 1) * BN, Nk);
    cp_async_commit();

    const int k0 = (j_begin + jj) * BN;
    const bool need_mask = (k0 + BN - 1 > tile_hi_min) || (k0 < tile_lo_max);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = q0 + ty * 4 + i;
      const int diag = row + off;
      const int hi_r = causal ? min(diag, Nk - 1) : Nk - 1;
      const int lo_r = window > 0 ? diag - window + 1 : 0;
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        float x = s[i][n] * c;
        if (need_mask) {
          const int key = k0 + tx + 16 * n;
          if (key > hi_r || key < lo_r) x = -CUDART_INF_F;
        }
        s[i][n] = x;
        mx = fmaxf(mx, x);
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m[i], mx);
      const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
      const float alpha = ex2_approx(m[i] - m_use);  // m = -inf -> 0
      m[i] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const float pv = ex2_approx(s[i][n] - m_use);
        sum += pv;
        Ps[(ty * 4 + i) * BN + tx + 16 * n] = pv;
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      l[i] = l[i] * alpha + sum;
      const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
      for (int d = 0; d < DP; ++d) acc[i][d] = f2_mul(acc[i][d], alpha2);
    }
    cp_async_wait<1>();
    __syncthreads();  // P tile complete; V_j visible

    // ---- O += P V: rows ty*4+i, columns tx*4.. (+64 for D = 128), or tx*2.. for D = 32
#pragma unroll 2
    for (int kk = 0; kk < BN; kk += 4) {
      float4 pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = *reinterpret_cast<const float4*>(Ps + (ty * 4 + i) * BN + kk);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float* vrow = Vs + (kk + u) * D;
        uint64_t vv[DP];   // pairs of adjacent columns
        if constexpr (DC == 8) {
          const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(vrow + tx * 4);
          const ulonglong2 bb = *reinterpret_cast<const ulonglong2*>(vrow + 64 + tx * 4);
          vv[0] = a.x; vv[1] = a.y; vv[2] = bb.x; vv[3] = bb.y;
        } else if constexpr (DC == 4) {
          const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(vrow + tx * 4);
          vv[0] = a.x; vv[1] = a.y;
        } else {
          vv[0] = *reinterpret_cast<const unsigned long long*>(vrow + tx * 2);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float pw = u == 0 ? pr[i].x : u == 1 ? pr[i].y : u == 2 ? pr[i].z : pr[i].w;
          const uint64_t pw2 = f2_pack(pw, pw);
#pragma unroll
          for (int d = 0; d < DP; ++d) acc[i][d] = f2_fma(pw2, vv[d], acc[i][d]);
        }
      }
    }
    __syncthreads();  // everyone is done with V_j: stream V_j+1 in during the next Q K^T
    if (jj + 1 < n_tiles) load_rows<D, false>(Vs, Vh, (j_begin + jj + 1) * BN, Nk);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // ---- epilogue
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = q0 + ty * 4 + i;
    if (row >= Nq) continue;
    const float inv_l = l[i] > 0.f ? 1.f / l[i] : 0.f;
    float* orow = O + ((static_cast<size_t>(b) * Hq + h) * Nq + row) * D;
    float a[DC];
#pragma unroll
    for (int d = 0; d < DP; ++d) {
      f2_unpack(acc[i][d], a[2 * d], a[2 * d + 1]);
      a[2 * d] *= inv_l;
      a[2 * d + 1] *= inv_l;
    }
    if constexpr (DC == 8) {
      *reinterpret_cast<float4*>(orow + tx * 4) = make_float4(a[0], a[1], a[2], a[3]);
      *reinterpret_cast<float4*>(orow + 64 + tx * 4) = make_float4(a[4], a[5], a[6], a[7]);
    } else if constexpr (DC == 4) {
      *reinterpret_cast<float4*>(orow + tx * 4) = make_float4(a[0], a[1], a[2], a[3]);
    } else {
      *reinterpret_cast<float2*>(orow + tx * 2) = make_float2(a[0], a[1]);
    }
    if (tx == 0 && LSE != nullptr)
      LSE[(static_cast<size_t>(b) * Hq + h) * Nq + row] =
          l[i] > 0.f ? (m[i] + log2f(l[i])) * 0.69314718055994531f : -CUDART_INF_F;
  }
}

template <int D>
int launch(const float* q, const float* k, const float* v, float* o, float* lse, int B, int Hq,
           int Hkv, int Nq, int Nk, float scale, int causal, int window, cudaStream_t stream) {
  static KernelSetup setup;
  if (const int rc = prepare_kernel(setup, attn_fwd_fp32_kernel<D>, Smem<D>::BYTES); rc != ATTN_OK) return rc;
  const dim3 grid((Nq + BM - 1) / BM, Hq, B);
  attn_fwd_fp32_kernel<D><<<grid, NT, Smem<D>::BYTES, stream>>>(
      q, k, v, o, lse, Hq, Hkv, Nq, Nk, scale * 1.4426950408889634f, causal, window > 0 ? window : 0);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace fwd_fp32

int launch_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                    int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
                    cudaStream_t stream, int* /*err*/) {
  switch (D) {
    case 32: return fwd_fp32::launch<32>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, stream);
    case 64: return fwd_fp32::launch<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, stream);
    case 128: return fwd_fp32::launch<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, stream);
    default: return ATTN_ERR_HEAD_DIM;
  }
}

}  // namespace attn

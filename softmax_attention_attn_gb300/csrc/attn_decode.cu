// attn_decode.cu — split-KV decode for sm_103a: partial step and combine step.
//
// Split-KV decode is one mode of the attention forward's feature surface in
// "Ask, Don't Equip: Question-Driven Coding Agents for Deep Kernel Optimization"
// (section "研究动机"); each chunk is the tiled online-softmax attention of
// "Agent 帮我写 CUDA：一个 Softmax Attention 算子的开发全记录" (section 四)
// restricted to the chunk's keys.  Chunks cover keys [c*chunk, (c+1)*chunk) of
// each sequence; the combine step weights chunk c by exp(LSE_c - max LSE).
//
// The partial step is bound by HBM bandwidth (about 2 flops per byte), so it
// uses no tensor cores.  Design:
//   * persistent CTAs walk a work list of (sequence b, chunk c, KV head) items,
//     built in shared memory from the device-side sequence lengths (no host
//     round trip); the KV heads of one chunk are adjacent items, so
//     neighbouring CTAs read neighbouring 256-byte rows of the cache;
//   * one producer thread streams 64-key K and V tiles ([64 keys][128] bf16,
//     16 KB, through a 3-slot TMA ring; or [64 keys][128] fp8 E4M3 codes,
//     8 KB, through a 6-slot ring), so 48 KB per CTA and, with three CTAs per
//     SM, 144 KB per SM are in flight (three CTAs rather than two with larger
//     rings: the consumers, not the copies, set the pace, and more resident
//     warps hide their latencies better);
//   * an fp8 cache holds E4M3 codes whose values are code * k_scale (K) and
//     code * v_scale (V): codes convert exactly to fp32 (through f16, which
//     holds every E4M3 value), k_scale folds into the softmax scale and v_scale
//     scales each chunk's output;
//   * four consumer warps: all G = Hq/Hkv query heads of the KV head share
//     each K/V tile.  For the scores, a thread multiplies 16 bytes of 8 key
//     rows by the G query slices it holds in registers and a 16-lane
//     reduce-scatter (halving exchange) finishes the dot products with about
//     one shuffle per score.  The chunk's softmax runs in shared memory in the
//     exp2 domain; P V accumulates per thread and is reduced across the eight
//     key groups through shared memory.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace decode {

constexpr int HD = 128;
constexpr int TILE = 64;                      // keys per TMA tile
constexpr int MAX_STAGES = 10;

// Residency and ring geometry for a bf16 (KV8 = false) or fp8 E4M3 (KV8 = true)
// cache: three CTAs per SM with 48 KB rings (144 KB in flight per SM); four with
// 32 KB rings (128 KB) for the fp8 cache with up to four query heads per KV
// head, whose consumers need the extra warps most and fit in the registers.
template <int G, bool KV8>
struct Ring {
  static constexpr int CTAS_PER_SM = (KV8 && G <= 4) ? 4 : 3;
  static constexpr int RING_BYTES = (CTAS_PER_SM == 4 ? 2 : 3) * TILE * HD * 2;
  static constexpr int ROW_BYTES = KV8 ? HD : 2 * HD;  // one key row of one KV head
  static constexpr int TILE_BYTES = TILE * ROW_BYTES;
  static constexpr int STAGES = RING_BYTES / TILE_BYTES;
  static_assert(STAGES <= MAX_STAGES, "ring slots");
};
constexpr int NCW = 4;                        // consumer warps
constexpr int NC = NCW * 32;                  // consumer threads
constexpr int NTHREADS = NC + 32;             // + producer warp

struct Layout {
  int ring, work, stats, bars, misc, split, bytes;
};

__host__ __device__ inline Layout layout(int G, int chunk, int B, int ring_bytes) {
  Layout L;
  L.ring = 0;
  L.work = L.ring + ring_bytes;
  const int scores = G * chunk * 4;
  const int red = 8 * G * HD * 4;
  L.stats = L.work + (scores > red ? scores : red);
  L.bars = L.stats + 2 * 8 * 4;                // m[8], l[8]
  L.misc = L.bars + 2 * MAX_STAGES * 8;
  L.split = L.misc + 16;                       // misc: abort flag, stop flag
  L.bytes = L.split + (B + 1) * 4;
  return L;
}

// 16-lane reduce-scatter: V partial sums per lane -> complete sums, R = max(V/16,1)
// per lane.  Lane g (0..15) ends with value indices g*R .. g*R+R-1 (V >= 16) or
// g/2 (V == 8, lane pairs hold the same value).
template <int V>
__device__ __forceinline__ void reduce_scatter16(float (&v)[V], int g) {
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int o = 8 >> st;
    const int n = V >> st;
    const bool hi = (g & o) != 0;
    if (n > 1) {
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float keep = hi ? v[i + n / 2] : v[i];
        const float send = hi ? v[i] : v[i + n / 2];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Eight E4M3 codes (the bytes of u, lowest first) to fp32.  Every E4M3 value
// is exact in f16, so the conversion is exact.
__device__ __forceinline__ void e4m3x8_to_float(const uint2& u, float (&f)[8]) {
  const uint32_t w[2] = {u.x, u.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t h01, h23;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(w[i]));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    f[4 * i + 0] = a.x;
    f[4 * i + 1] = a.y;
    f[4 * i + 2] = b.x;
    f[4 * i + 3] = b.y;
  }
}

// The 8 elements [g16 * 8, g16 * 8 + 8) of key row `key` of a ring tile, as fp32.
template <bool KV8>
__device__ __forceinline__ void row_slice(const uint8_t* tile, int key, int g16, float (&f)[8]) {
  if constexpr (KV8) {
    e4m3x8_to_float(*reinterpret_cast<const uint2*>(tile + key * HD + g16 * 8), f);
  } else {
    bf16x8_to_float(*reinterpret_cast<const uint4*>(tile + key * (HD * 2) + g16 * 16), f);
  }
}

// acc[h][e] += sum over the 8 keys (ksub + 8 i) of one 64-key tile of
// p[h][key] * v[key][g16 * 8 + e].  With MASK, keys >= valid contribute 0.
template <int G, bool MASK, bool KV8>
__device__ __forceinline__ void pv_tile(float (&acc)[G][8], const uint8_t* tile, const float* pt,
                                        int chunk, int ksub, int g16, int valid) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int key = ksub + 8 * i;
    float vf[8];
    row_slice<KV8>(tile, key, g16, vf);
    if (MASK && key >= valid) {
#pragma unroll
      for (int e = 0; e < 8; ++e) vf[e] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float pw = pt[h * chunk + key];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pw, vf[e], acc[h][e]);
    }
  }
}

struct Work {
  int b, c, kvh, n_valid, ntl;
};

__device__ __forceinline__ Work decode_work(int w, const int* split, int B, int Hkv, int chunk,
                                            const int* __restrict__ seqlens) {
  Work r;
  const int gc = w / Hkv;
  r.kvh = w - gc * Hkv;
  int lo = 0, hi = B;  // largest b with split[b] <= gc
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (split[mid] <= gc) lo = mid; else hi = mid;
  }
  r.b = lo;
  r.c = gc - split[lo];
  const int L = __ldg(seqlens + lo);
  r.n_valid = min(chunk, L - r.c * chunk);
  r.ntl = (r.n_valid + TILE - 1) / TILE;
  return r;
}

// Paged cache: key j of sequence b is row j % page_size of page
// block_table[b * max_pages + j / page_size] of a page pool [num_pages,
// page_size, Hkv, D]; page_size is a multiple of the 64-key tile, so a tile
// never straddles two pages.
struct Paging {
  const int* block_table;
  int max_pages, page_size, num_pages;
};

template <int G, bool PAGED, bool KV8>
__global__ void __launch_bounds__(NTHREADS, (Ring<G, KV8>::CTAS_PER_SM))
attn_decode_splitkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __nv_bfloat16* __restrict__ q, const int* __restrict__ seqlens,
                           float* __restrict__ ws_o, float* __restrict__ ws_lse, int B, int Hq,
                           int Hkv, int Nk_max, int chunk, int S_max, float c_log2, float v_scale,
                           int* err, const Paging pg) {
  constexpr int STAGES = Ring<G, KV8>::STAGES;
  constexpr int TILE_BYTES = Ring<G, KV8>::TILE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const Layout L = layout(G, chunk, B, Ring<G, KV8>::RING_BYTES);
  float* work = reinterpret_cast<float*>(smem + L.work);   // scores / p, then reduction buffer
  float* st_m = reinterpret_cast<float*>(smem + L.stats);
  float* st_l = st_m + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
  int* split = reinterpret_cast<int*>(smem + L.split);
  auto bar_full = [&](int s) { return sb + L.bars + 8u * s; };
  auto bar_empty = [&](int s) { return sb + L.bars + 8u * (STAGES + s); };

  const int warp = warp_id_uniform();
  const int lane = static_cast<int>(lane_id());
  const int tid = static_cast<int>(threadIdx.x);

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), NCW);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  // ---- work list: split[b] = number of chunks of sequences 0..b-1 (one warp)
  if (warp == 0) {
    const int per = (B + 31) / 32;
    const int b0 = min(B, lane * per), b1 = min(B, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      const int Lb = seqlens[b];
      if (Lb < 1 || Lb > Nk_max) {
        atomicCAS(err, 0, ATTN_ERR_SEQLEN);
        continue;
      }
      local += (Lb + chunk - 1) / chunk;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int b = b0; b < b1; ++b) {
      split[b] = run;
      const int Lb = seqlens[b];
      if (Lb >= 1 && Lb <= Nk_max) run += (Lb + chunk - 1) / chunk;
    }
    if (lane == 31) split[B] = incl;
  }
  __syncthreads();
  const int total = split[B] * Hkv;

  if (warp == NCW) {
    // ================================================================ producer
    if (lane == 0) {
      int it = 0;
      int cached_lp = -1, cached_b = -1, cached_page = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const Work wk = decode_work(w, split, B, Hkv, chunk, seqlens);
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const CUtensorMap* m = kv ? &tm_v : &tm_k;
          for (int tl = 0; tl < wk.ntl; ++tl, ++it) {
            const int s = it % STAGES, u = it / STAGES;
            if (u > 0 && !mbar_wait(bar_empty(s), (u - 1) & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar_full(s), TILE_BYTES);
            const int key0 = wk.c * chunk + tl * TILE;
            if constexpr (PAGED) {
              const int lp = key0 / pg.page_size;
              if (lp != cached_lp || wk.b != cached_b) {  // one block-table read per page
                cached_page = __ldg(pg.block_table + static_cast<size_t>(wk.b) * pg.max_pages + lp);
                cached_lp = lp;
                cached_b = wk.b;
              }
              int page = cached_page;
              if (page < 0 || page >= pg.num_pages) {  // reported; the copy reads zeros instead
                atomicCAS(err, 0, ATTN_ERR_PAGE);
                page = pg.num_pages;
              }
              tma_load_4d(sb + L.ring + s * TILE_BYTES, m, bar_full(s), 0, wk.kvh,
                          key0 - lp * pg.page_size, page);
            } else {
              tma_load_4d(sb + L.ring + s * TILE_BYTES, m, bar_full(s), 0, wk.kvh, key0, wk.b);
            }
          }
        }
      }
      if (!ok) {
        for (int i = max(0, it - STAGES); i < it; ++i) {
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(bar_full(i % STAGES), (i / STAGES) & 1))
            if (global_ns() - t0 > kAttnWaitNs) break;
        }
      }
    }
    return;
  }

  // ==================================================================== consumers
  // A failed (timed-out) wait never breaks out of the item early: every
  // consumer keeps reaching the same named barriers, and the decision to stop
  // is taken at the end of the item from one shared copy of the abort flag.
  volatile int* stop = abort_flag + 1;
  const int g16 = tid & 15;       // 16-byte column slice of a 256-byte row
  const int ksub = tid >> 4;      // key sub-group 0..7
  constexpr int V = 8 * G;        // partial sums per thread per tile
  constexpr int R = V >= 16 ? V / 16 : 1;
  int it = 0;
  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const Work wk = decode_work(w, split, B, Hkv, chunk, seqlens);
    const int h0 = wk.kvh * G;
    float qr[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(q + (static_cast<size_t>(wk.b) * Hq + h0 + h) * HD) + g16);
      bf16x8_to_float(u, qr[h]);
    }
    // ---- phase 1: scores s[h][key] = q_h . k_key
    bool ok = true;
    for (int tl = 0; tl < wk.ntl; ++tl, ++it) {
      const int s = it % STAGES;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_full(s), (it / STAGES) & 1, abort_flag, err));
      if (!ok) continue;
      const uint8_t* tile = smem + L.ring + s * TILE_BYTES;
      float v[V];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int key = ksub + 8 * i;
        float kf[8];
        row_slice<KV8>(tile, key, g16, kf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaf(qr[h][e], kf[e], a);
          v[i * G + h] = a;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty(s));
      reduce_scatter16<V>(v, g16);
      if (V >= 16 || (g16 & 1) == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int idx = V >= 16 ? g16 * R + r : (g16 >> 1);
          const int i = idx / G, h = idx % G;
          const int key = tl * TILE + ksub + 8 * i;
          work[h * chunk + key] = key < wk.n_valid ? v[r] : -CUDART_INF_F;
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
    // ---- phase 2: chunk softmax per head (exp2 domain), p written in place
    const int nk_pad = wk.ntl * TILE;
    for (int h = warp; h < G; h += NCW) {
      float* sh = work + h * chunk;
      float mx = -CUDART_INF_F;
      for (int j = lane; j < nk_pad; j += 32) mx = fmaxf(mx, sh[j]);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m = (mx == -CUDART_INF_F) ? 0.f : mx * c_log2;
      float sum = 0.f;
      for (int j = lane; j < nk_pad; j += 32) {
        const float pv = ex2_approx(fmaf(sh[j], c_log2, -m));
        sh[j] = pv;
        sum += pv;
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        st_m[h] = m;
        st_l[h] = sum;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
    // ---- phase 3: O = sum_key p[h][key] v_key
    float acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    for (int tl = 0; tl < wk.ntl; ++tl, ++it) {
      const int s = it % STAGES;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_full(s), (it / STAGES) & 1, abort_flag, err));
      if (!ok) continue;
      const uint8_t* tile = smem + L.ring + s * TILE_BYTES;
      const float* pt = work + tl * TILE;
      // Only a chunk's last tile can reach past the sequence: that tile takes the
      // masked copy of the loop, which zeroes the extra rows (p is 0 there, but
      // 0 * NaN from an unused cache row is not).
      const int valid_here = wk.n_valid - tl * TILE;
      if (valid_here >= TILE)
        pv_tile<G, false, KV8>(acc, tile, pt, chunk, ksub, g16, TILE);
      else
        pv_tile<G, true, KV8>(acc, tile, pt, chunk, ksub, g16, valid_here);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty(s));
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");  // p no longer needed
    float* red = work;                                      // [8][G][HD]
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float4* dst = reinterpret_cast<float4*>(red + (ksub * G + h) * HD + g16 * 8);
      dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
    {
      const int d = tid;  // 0..127
      const size_t base = (static_cast<size_t>(wk.b) * Hq + h0) * S_max + wk.c;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) o += red[(k * G + h) * HD + d];
        ws_o[(base + static_cast<size_t>(h) * S_max) * HD + d] = o / st_l[h] * v_scale;
      }
      if (tid < G) ws_lse[base + static_cast<size_t>(tid) * S_max] = (st_m[tid] + log2f(st_l[tid])) * 0.69314718055994531f;
      if (tid == 0) *stop = *abort_flag;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");  // red free for the next item
    if (*stop) break;
  }
}

// One warp per (b, h): LSE-weighted merge of the chunk results.
__global__ void __launch_bounds__(128)
attn_decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                           const int* __restrict__ seqlens, __nv_bfloat16* __restrict__ o,
                           float* __restrict__ lse, int B, int Hq, int Nk_max, int chunk, int S_max,
                           int* err) {
  const int lane = static_cast<int>(lane_id());
  const int bh = static_cast<int>(blockIdx.x) * 4 + static_cast<int>(threadIdx.x >> 5);
  if (bh >= B * Hq) return;
  const int b = bh / Hq;
  const int Lb = __ldg(seqlens + b);
  __nv_bfloat16* orow = o + static_cast<size_t>(bh) * HD + lane * 4;
  if (Lb < 1 || Lb > Nk_max) {
    if (lane == 0) atomicCAS(err, 0, ATTN_ERR_SEQLEN);
    *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
    if (lane == 0 && lse != nullptr) lse[bh] = -CUDART_INF_F;
    return;
  }
  const int n = (Lb + chunk - 1) / chunk;
  const float* lp = ws_lse + static_cast<size_t>(bh) * S_max;
  const float* op = ws_o + static_cast<size_t>(bh) * S_max * HD + lane * 4;
  float M = -CUDART_INF_F;
  for (int c = lane; c < n; c += 32) M = fmaxf(M, lp[c]);
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, k));
  constexpr float LOG2E = 1.4426950408889634f;
  float s = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < n; c0 += 32) {
    const float wc = (c0 + lane < n) ? ex2_approx((lp[c0 + lane] - M) * LOG2E) : 0.f;
    s += wc;
    const int cnt = min(32, n - c0);
    // eight chunks at a time, all eight loads in flight before the sums (chunks past the
    // count load zeros and add nothing: their weights are finite)
    for (int j0 = 0; j0 < cnt; j0 += 8) {
      float4 x[8];
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        w[u] = __shfl_sync(0xffffffffu, wc, j & 31);
        x[u] = j < cnt ? *reinterpret_cast<const float4*>(op + static_cast<size_t>(c0 + j) * HD)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x = fmaf(w[u], x[u].x, acc.x);
        acc.y = fmaf(w[u], x[u].y, acc.y);
        acc.z = fmaf(w[u], x[u].z, acc.z);
        acc.w = fmaf(w[u], x[u].w, acc.w);
      }
    }
  }
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
  const float inv = 1.f / s;
  *reinterpret_cast<uint2*>(orow) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (lane == 0 && lse != nullptr) lse[bh] = M + logf(s);
}

template <int G, bool PAGED, bool KV8>
int launch_split(const CUtensorMap& tk, const CUtensorMap& tv, const void* q, const int* seqlens,
                 float* ws_o, float* ws_lse, int B, int Hq, int Hkv, int Nk_max, float scale,
                 int chunk, int S_max, int num_sms, cudaStream_t stream, int* err, const Paging& pg,
                 float k_scale, float v_scale) {
  const Layout L = layout(G, chunk, B, Ring<G, KV8>::RING_BYTES);
  const int smem = L.bytes + 1024;
  static int attr_dev = -1;
  static int attr_bytes = 0;
  static int attr_smem = -1;   // shared-memory size the resident count below is for
  static int resident = 1;     // CTAs of this instance that fit on one SM
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev || attr_bytes < smem) {
    if (cudaFuncSetAttribute(attn_decode_splitkv_kernel<G, PAGED, KV8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_dev = dev;
    attr_bytes = smem;
    attr_smem = -1;
  }
  if (attr_smem != smem) {
    // the persistent grid is as many CTAs as are resident at once: up to three
    // (fp8 cache, G <= 4: four) per SM, fewer when a large chunk or head group
    // enlarges the score area
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_splitkv_kernel<G, PAGED, KV8>, NTHREADS,
                                                      smem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    constexpr int cap = Ring<G, KV8>::CTAS_PER_SM;
    resident = n < 1 ? 1 : (n > cap ? cap : n);
    attr_smem = smem;
  }
  const int grid = resident * num_sms;
  attn_decode_splitkv_kernel<G, PAGED, KV8><<<grid, NTHREADS, smem, stream>>>(
      tk, tv, static_cast<const __nv_bfloat16*>(q), seqlens, ws_o, ws_lse, B, Hq, Hkv, Nk_max, chunk,
      S_max, scale * k_scale * 1.4426950408889634f, v_scale, err, pg);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <bool PAGED, bool KV8>
int launch_split_any(const CUtensorMap& tk, const CUtensorMap& tv, const void* q, const int* seqlens,
                     void* workspace, int B, int Hq, int Hkv, int Nk_max, float scale, int chunk,
                     int num_sms, cudaStream_t stream, int* err, const Paging& pg, float k_scale,
                     float v_scale) {
  const int S_max = (Nk_max + chunk - 1) / chunk;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_lse = ws_o + static_cast<size_t>(B) * Hq * S_max * HD;
#define ATTN_SPLIT_ARGS tk, tv, q, seqlens, ws_o, ws_lse, B, Hq, Hkv, Nk_max, scale, chunk, S_max, \
                        num_sms, stream, err, pg, k_scale, v_scale
  switch (Hq / Hkv) {
    case 1: return launch_split<1, PAGED, KV8>(ATTN_SPLIT_ARGS);
    case 2: return launch_split<2, PAGED, KV8>(ATTN_SPLIT_ARGS);
    case 4: return launch_split<4, PAGED, KV8>(ATTN_SPLIT_ARGS);
    case 8: return launch_split<8, PAGED, KV8>(ATTN_SPLIT_ARGS);
    default: return ATTN_ERR_GQA;
  }
#undef ATTN_SPLIT_ARGS
}

// Tensor maps over a contiguous cache [B, Nk_max, Hkv, D] or a page pool
// [num_pages, page_size, Hkv, D]: one box is 64 key rows of one KV head.
inline bool cache_maps(CUtensorMap* tk, CUtensorMap* tv, const void* k, const void* v, int Hkv,
                       int rows, int outer, bool kv8) {
  const uint32_t box[4] = {HD, 1, TILE, 1};
  const CUtensorMapDataType dt = kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t es = kv8 ? 1 : 2;
  return encode_tiled_4d(tk, dt, k, HD, Hkv, rows, outer, es, box, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode_tiled_4d(tv, dt, v, HD, Hkv, rows, outer, es, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace decode

int launch_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                          const int* seqlens, void* workspace, int B, int Hq, int Hkv,
                          int Nk_max, float scale, int chunk, int num_sms, cudaStream_t stream,
                          int* err, int kv8, float k_scale, float v_scale) {
  using namespace decode;
  CUtensorMap tk, tv;
  if (!cache_maps(&tk, &tv, k_cache, v_cache, Hkv, Nk_max, B, kv8 != 0)) return ATTN_ERR_CUDA;
  const Paging none{nullptr, 0, 0, 0};
  return kv8 ? launch_split_any<false, true>(tk, tv, q, seqlens, workspace, B, Hq, Hkv, Nk_max, scale,
                                             chunk, num_sms, stream, err, none, k_scale, v_scale)
             : launch_split_any<false, false>(tk, tv, q, seqlens, workspace, B, Hq, Hkv, Nk_max, scale,
                                              chunk, num_sms, stream, err, none, 1.f, 1.f);
}

int launch_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int* block_table, const int* seqlens, void* workspace, int B,
                                int Hq, int Hkv, int num_pages, int page_size, int max_pages,
                                float scale, int chunk, int num_sms, cudaStream_t stream, int* err,
                                int kv8, float k_scale, float v_scale) {
  using namespace decode;
  CUtensorMap tk, tv;
  if (!cache_maps(&tk, &tv, k_pages, v_pages, Hkv, page_size, num_pages, kv8 != 0)) return ATTN_ERR_CUDA;
  const Paging pg{block_table, max_pages, page_size, num_pages};
  return kv8 ? launch_split_any<true, true>(tk, tv, q, seqlens, workspace, B, Hq, Hkv,
                                            max_pages * page_size, scale, chunk, num_sms, stream, err,
                                            pg, k_scale, v_scale)
             : launch_split_any<true, false>(tk, tv, q, seqlens, workspace, B, Hq, Hkv,
                                             max_pages * page_size, scale, chunk, num_sms, stream, err,
                                             pg, 1.f, 1.f);
}

int launch_decode_combine(const void* workspace, const int* seqlens, void* o, float* lse, int B,
                          int Hq, int Nk_max, int chunk, cudaStream_t stream, int* err) {
  using namespace decode;
  const int S_max = (Nk_max + chunk - 1) / chunk;
  const float* ws_o = static_cast<const float*>(workspace);
  const float* ws_lse = ws_o + static_cast<size_t>(B) * Hq * S_max * HD;
  const int grid = (B * Hq + 3) / 4;
  attn_decode_combine_kernel<<<grid, 128, 0, stream>>>(ws_o, ws_lse, seqlens,
                                                        static_cast<__nv_bfloat16*>(o), lse, B, Hq,
                                                        Nk_max, chunk, S_max, err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

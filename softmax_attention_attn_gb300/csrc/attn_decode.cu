// attn_decode.cu — split-KV decode for sm_103a: partial step and combine step.
//
// Split-KV decode is one mode of the attention forward's feature surface in
// "Ask, Don't Equip: Question-Driven Coding Agents for Deep Kernel Optimization"
// (section "研究动机"); each chunk is the tiled online-softmax attention of
// "Agent 帮我写 CUDA：一个 Softmax Attention 算子的开发全记录" (section 四)
// restricted to the chunk's keys.  Chunks cover keys [c*chunk, (c+1)*chunk) of
// each sequence; the combine step weights chunk c by exp(LSE_c - max LSE).
//
// The partial step should be bound by HBM bandwidth.  Two consumers serve it:
//
// SIMT consumer (bf16 cache, head dimension 128, up to 8 query heads per KV
// head: about 2-8 FLOP per byte, within what the FP32 pipes do at HBM speed):
//   * persistent CTAs walk a work list of (sequence b, chunk c, KV head) items,
//     built in shared memory from the device-side sequence lengths (no host
//     round trip); the KV heads of one chunk are adjacent items, so
//     neighbouring CTAs read neighbouring 256-byte rows of the cache;
//   * one producer thread streams 64-key K and V tiles ([64 keys][128] bf16,
//     16 KB) through a 3-slot TMA ring, so 48 KB per CTA and, with three CTAs
//     per SM, 144 KB per SM are in flight (three CTAs rather than two with
//     larger rings: the consumers, not the copies, set the pace, and more
//     resident warps hide their latencies better);
//   * four consumer warps: all G = Hq/Hkv query heads of the KV head share
//     each K/V tile.  For the scores, a thread multiplies 16 bytes of 8 key
//     rows by the G query slices it holds in registers and a 16-lane
//     reduce-scatter (halving exchange) finishes the dot products with about
//     one shuffle per score.  The chunk's softmax runs in shared memory in the
//     exp2 domain; P V accumulates per thread and is reduced across the eight
//     key groups through shared memory.
//
// Tensor-core consumer (fp8 E4M3 cache, head dimension 64, 16 or 32 query heads
// per KV head): the same work list, producer and chunk softmax, with the two
// products on warp-level MMAs; see the section "tensor-core partial step".
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace decode {

constexpr int HD = 128;
constexpr int TILE = 64;                      // keys per TMA tile
constexpr int MAX_STAGES = 10;

// Residency and ring geometry of the SIMT consumer (bf16 cache): three CTAs per
// SM with 48 KB rings (144 KB in flight per SM).
template <int G>
struct Ring {
  static constexpr int CTAS_PER_SM = 3;
  static constexpr int RING_BYTES = 3 * TILE * HD * 2;
  static constexpr int ROW_BYTES = 2 * HD;             // one key row of one KV head
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

// The 8 elements [g16 * 8, g16 * 8 + 8) of key row `key` of a ring tile, as fp32.
__device__ __forceinline__ void row_slice(const uint8_t* tile, int key, int g16, float (&f)[8]) {
  bf16x8_to_float(*reinterpret_cast<const uint4*>(tile + key * (HD * 2) + g16 * 16), f);
}

// acc[h][e] += sum over the 8 keys (ksub + 8 i) of one 64-key tile of
// p[h][key] * v[key][g16 * 8 + e].  With MASK, keys >= valid contribute 0.
template <int G, bool MASK>
__device__ __forceinline__ void pv_tile(float (&acc)[G][8], const uint8_t* tile, const float* pt,
                                        int chunk, int ksub, int g16, int valid) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int key = ksub + 8 * i;
    float vf[8];
    row_slice(tile, key, g16, vf);
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

template <int G, bool PAGED>
__global__ void __launch_bounds__(NTHREADS, (Ring<G>::CTAS_PER_SM))
attn_decode_splitkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __nv_bfloat16* __restrict__ q, const int* __restrict__ seqlens,
                           float* __restrict__ ws_o, float* __restrict__ ws_lse, int B, int Hq,
                           int Hkv, int Nk_max, int chunk, int S_max, float c_log2, int* err,
                           const Paging pg) {
  constexpr int STAGES = Ring<G>::STAGES;
  constexpr int TILE_BYTES = Ring<G>::TILE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const Layout L = layout(G, chunk, B, Ring<G>::RING_BYTES);
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
      const uint64_t stream_policy = l2_policy_evict_first();   // the cache is read once
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
              tma_load_4d_hint(sb + L.ring + s * TILE_BYTES, m, bar_full(s), 0, wk.kvh,
                               key0 - lp * pg.page_size, page, stream_policy);
            } else {
              tma_load_4d_hint(sb + L.ring + s * TILE_BYTES, m, bar_full(s), 0, wk.kvh, key0, wk.b, stream_policy);
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
  // chunk results: kept in L2 for the combine step, which reads them right after this kernel
  const uint64_t keep_policy = l2_policy_evict_last();
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
        row_slice(tile, key, g16, kf);
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
        pv_tile<G, false>(acc, tile, pt, chunk, ksub, g16, TILE);
      else
        pv_tile<G, true>(acc, tile, pt, chunk, ksub, g16, valid_here);
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
        st_global_hint(ws_o + (base + static_cast<size_t>(h) * S_max) * HD + d, o / st_l[h], keep_policy);
      }
      if (tid < G)
        st_global_hint(ws_lse + base + static_cast<size_t>(tid) * S_max,
                       (st_m[tid] + log2f(st_l[tid])) * 0.69314718055994531f, keep_policy);
      if (tid == 0) *stop = *abort_flag;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");  // red free for the next item
    if (*stop) break;
  }
}

// ====================================================================== tensor-core partial step
// The same partial step for an fp8 (E4M3) cache, for head dimension 64, and for
// 16 or 32 query heads per KV head.  There the SIMT consumers above cannot keep
// up with HBM: an fp8 byte needs its conversion plus G multiply-adds for Q K and
// again for P V (about 16 FLOP per byte at G = 4), and G = 16 or 32 query heads
// per KV head need 16-32 FLOP per byte of a bf16 cache, both above what the FP32
// pipes deliver per byte of HBM bandwidth.  Both products of a chunk are small
// dense contractions (G x D x 64 keys per tile), so the consumer warps run them
// as warp-level tensor-core MMAs (m16n8k16, fp32 accumulation):
//   * Q K^T: a warp takes 16 keys of a tile; the A operand is the K rows,
//     read from the 128-byte (64-byte for 64-byte rows) swizzled TMA tile and,
//     for fp8, converted in registers (cvt.rn.f16x2.e4m3x2, exact: every E4M3
//     value is an f16 value); the B operand is Q^T in registers (8 query heads per
//     MMA column block).  Thread (g, c) of a warp supplies the head-dimension
//     slice [c D/4, (c+1) D/4) in every K step (the sum over d may visit d in
//     any order, so the MMA's K index is permuted to make that slice contiguous).
//   * For an fp8 cache the MMAs run on f16 operands: each query head is scaled
//     by a power of two into f16 range (exact) and its scores are scaled back.
//   * P V: O^T = V^T P^T; warp w owns the head-dimension rows [w D/4, (w+1) D/4)
//     and reads V^T fragments from the tile (pairs of keys at one d are gathered
//     with byte permutes); P is read from the chunk's score rows in shared
//     memory and rounded to the MMA operand type (f16 for fp8, else bf16).  No
//     reduction across warps is needed.
// Keys past a sequence's end get score -inf and V = 0 (an unused cache row may
// hold NaN, and 0 * NaN is NaN).
namespace decode_mma {

constexpr int TILE = 64;                 // keys per TMA tile
// floats of padding per score row (row stride chunk + SPAD, chunk a multiple of 64): a
// stride of 4 mod 32 words puts the score stores of Q K^T (heads 2c + e, keys g) and the
// 32-bit p loads of P V (heads g, key pairs c) on 32 different banks
constexpr int SPAD = 4;
constexpr int MAX_STAGES = 16;

template <int HD, bool KV8>
struct Geo {
  static constexpr int ESZ = KV8 ? 1 : 2;
  static constexpr int ROW = HD * ESZ;                  // bytes of one key row of one KV head
  static constexpr int SROW = ROW > 128 ? 128 : ROW;    // bytes of that row inside one swizzled slab
  static constexpr int SLABS = ROW / SROW;              // 2 for bf16 D = 128, else 1
  static constexpr int SLAB_BYTES = TILE * SROW;
  static constexpr int TILE_BYTES = TILE * ROW;
};

// Residency: up to 8 query heads per KV head, three (bf16) or four (fp8) CTAs per SM
// with 48 / 40 KB rings; with 16 or 32 the chunk's scores take 32-64 KB (chunk 512),
// so two CTAs share an SM with the ring slots the rest of half the shared memory holds
// (one CTA with up to 16 tiles when two do not fit).  The launch bound lets the
// compiler keep the registers within that residency.
// Consumer warps: four (warp w: keys [16w, 16w+16) of a tile in Q K^T, head-dimension rows
// [w D/4, (w+1) D/4) in P V) up to 8 query heads per KV head; eight with 16 or 32, where the
// products are long enough per item that a CTA alone on its SM needs more warps in flight
// (warp w then takes keys [16 (w % 4), +16) and half of the heads' MMA column blocks in Q K^T,
// and its share of the (head-dimension block, head column block) pairs in P V).
template <int HD, int G, bool KV8>
struct Cfg {
  static constexpr int NT = (G + 7) / 8;                // MMA column blocks of 8 query heads
  // up to 8 heads: four CTAs per SM with 40 KB rings for fp8 caches (the consumers' per-byte
  // work needs the warps), three with 48 KB rings for bf16 (measured: fp8 5422 -> 5560 GB/s with
  // four; bf16 D = 64 6030 -> 5560 with four); 16 or 32 heads: two
  static constexpr int CTAS_PER_SM = G <= 8 ? (KV8 ? 4 : 3) : 2;
  static constexpr int SMALL_RING_BYTES = (KV8 ? 40 : 48) * 1024;    // G <= 8
  static constexpr int NCW = G >= 16 ? 8 : 4;           // consumer warps
  static constexpr int NC = NCW * 32;
  static constexpr int NTHREADS = NC + 32;              // + producer warp
  // Q K^T: warp w takes key block w % 4 and column blocks [(w / 4) NTW, + NTW)
  static constexpr int NTW = NT / (NCW / 4);
  // P V: MB blocks of 16 head-dimension rows; a warp takes MTW consecutive blocks and
  // NTP column blocks
  static constexpr int MB = HD / 16;
  static constexpr int MTW = MB > NCW ? MB / NCW : 1;
  static constexpr int WPM = NCW > MB ? NCW / MB : 1;   // warps per block of rows
  static constexpr int NTP = NT / WPM;
  static_assert(NTW >= 1 && NTP >= 1 && NTW * (NCW / 4) == NT && NTP * WPM == NT, "warp split");
};

struct Layout {
  int work, stats, bars, misc, split, bytes;
};

__host__ __device__ inline Layout layout(int G, int chunk, int B, int ring_bytes) {
  Layout L;
  L.work = ring_bytes;                                  // scores, then p: [G][chunk + SPAD] fp32
  L.stats = L.work + G * (chunk + SPAD) * 4;
  L.bars = L.stats + 2 * 32 * 4;                        // m[32], l[32]
  L.misc = L.bars + 2 * MAX_STAGES * 8;
  L.split = L.misc + 16;                                // misc: abort flag, stop flag
  L.bytes = L.split + (B + 1) * 4;
  return L;
}

// Byte offset inside a ring tile of byte `b` of key row `row`: the row is split
// into slabs of SROW bytes, each slab a [64][SROW] block written by one TMA box
// with the 128-byte (SROW = 128) or 64-byte (SROW = 64) swizzle: the 16-byte
// chunk index is XORed with row & 7, respectively (row >> 1) & 3.
template <int HD, bool KV8>
__device__ __forceinline__ uint32_t tile_off(int row, int b) {
  using GE = Geo<HD, KV8>;
  const int slab = b / GE::SROW;
  const int bb = b % GE::SROW;
  int ch = bb >> 4;
  if constexpr (GE::SROW == 128) ch ^= row & 7;
  else ch ^= (row >> 1) & 3;
  return static_cast<uint32_t>(slab * GE::SLAB_BYTES + row * GE::SROW + (ch << 4) + (bb & 15));
}

// Two E4M3 codes (bits 0-15 of `w` if !HI, else bits 16-31) -> f16x2 (exact).
template <bool HI>
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t w) {
  uint32_t h;
  if constexpr (HI)
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(h) : "r"(w));
  else
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(h) : "r"(w));
  return h;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// D (16x8 fp32) += A (16x16) B (16x8): f16 operands if F16, else bf16.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int HD, int G, bool PAGED, bool KV8>
__global__ void __launch_bounds__(Cfg<HD, G, KV8>::NTHREADS, Cfg<HD, G, KV8>::CTAS_PER_SM)
attn_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __nv_bfloat16* __restrict__ q, const int* __restrict__ seqlens,
                       float* __restrict__ ws_o, float* __restrict__ ws_lse, int B, int Hq, int Hkv,
                       int Nk_max, int chunk, int S_max, float c_log2, float v_scale, int* err,
                       const decode::Paging pg, int STAGES) {
  using GE = Geo<HD, KV8>;
  using C = Cfg<HD, G, KV8>;
  constexpr int NCW = C::NCW;
  constexpr int NC = C::NC;
  constexpr int NTW = C::NTW;
  constexpr int NTP = C::NTP;
  constexpr int TILE_BYTES = GE::TILE_BYTES;
  constexpr int KK = HD / 16;             // K steps of Q K^T
  constexpr int DQ = HD / 4;              // head-dimension elements per thread in Q K^T
  constexpr int QW = DQ / 2;              // 32-bit words of 16-bit values per thread and head
  constexpr int KW = DQ * GE::ESZ / 4;    // 32-bit words of one K row slice per thread
  constexpr int MT = C::MTW;              // 16-row blocks of the head dimension per warp in P V
  constexpr int DV = 2 * MT;              // head-dimension elements per thread in P V
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const Layout L = layout(G, chunk, B, STAGES * TILE_BYTES);
  const int wstride = chunk + SPAD;
  float* work = reinterpret_cast<float*>(smem + L.work);
  float* st_m = reinterpret_cast<float*>(smem + L.stats);
  float* st_l = st_m + 32;
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
      // the cache is read once; 128-byte rows keep the default policy (neighbouring KV heads'
      // rows share DRAM bursts that L2 serves to the CTAs reading them)
      const uint64_t stream_policy = GE::ROW >= 256 ? l2_policy_evict_first() : l2_policy_evict_normal();
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const decode::Work wk = decode::decode_work(w, split, B, Hkv, chunk, seqlens);
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
            int row = key0, outer = wk.b;
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
              row = key0 - lp * pg.page_size;
              outer = page;
            }
#pragma unroll
            for (int sl = 0; sl < GE::SLABS; ++sl)
              tma_load_4d_hint(sb + s * TILE_BYTES + sl * GE::SLAB_BYTES, m, bar_full(s),
                               sl * (GE::SROW / GE::ESZ), wk.kvh, row, outer, stream_policy);
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
  // As in the SIMT consumer: a failed wait never leaves an item early; every
  // consumer reaches the same named barriers and the stop decision is taken at
  // the end of the item from one shared copy of the abort flag.
  volatile int* stop = abort_flag + 1;
  // chunk results: kept in L2 for the combine step, which reads them right after this kernel
  const uint64_t keep_policy = l2_policy_evict_last();
  const int g = lane >> 2;        // MMA row group
  const int c = lane & 3;         // thread in group
  const int kblk = warp & 3;      // Q K^T: key block of the tile
  const int nt0 = (warp >> 2) * NTW;                         // Q K^T: first column block
  const int mblk = warp % (C::MB / MT);                      // P V: first row block (of MT)
  const int pt0 = (warp / (C::MB / MT)) * NTP;               // P V: first column block
  int it = 0;
  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const decode::Work wk = decode::decode_work(w, split, B, Hkv, chunk, seqlens);
    const int h0 = wk.kvh * G;
    // bf16 D = 128: threads c >= 2 visit the 16-byte chunks of their slice in the
    // order 2, 3, 0, 1 (for K and, identically, for Q), so that the K loads of
    // threads c and c + 2, which read different slabs, fall into different banks
    const int rot = (GE::ROW == 256) ? 2 * (c >> 1) : 0;
    // ---- Q^T fragments: thread (g, c) holds head 8 (nt0 + nt) + g, elements [c DQ, (c+1) DQ)
    uint32_t qf[NTW][QW];
    float qsc[NTW][2];            // fp8 cache: the score scales of heads 8 (nt0 + nt) + 2c, + 1
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      const int h = 8 * (nt0 + nt) + g;
      uint32_t raw[QW];
      if (h < G) {
        const uint4* src = reinterpret_cast<const uint4*>(q + (static_cast<size_t>(wk.b) * Hq + h0 + h) * HD + c * DQ);
#pragma unroll
        for (int i = 0; i < QW / 4; ++i) {
          const uint4 u = __ldg(src + (i ^ rot));
          raw[4 * i + 0] = u.x;
          raw[4 * i + 1] = u.y;
          raw[4 * i + 2] = u.z;
          raw[4 * i + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < QW; ++i) raw[i] = 0u;
      }
      if constexpr (KV8) {
        // f16 operands: scale head h by 2^-e with e = floor(log2 max|q_h|) - 14, so that
        // the largest |q| lies in [2^14, 2^15) (exact: a power of two; bf16 values then
        // fit f16's 11-bit significand); the head's scores are multiplied by 2^e.
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < QW; ++i)
          amax = fmax3(amax, fabsf(__uint_as_float(raw[i] << 16)), fabsf(__uint_as_float(raw[i] & 0xFFFF0000u)));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int e = 0;
        if (amax > 0.f) e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14;
        e = max(-100, min(100, e));
        const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
        for (int i = 0; i < QW; ++i)
          qf[nt][i] = pack_f16x2(__uint_as_float(raw[i] << 16) * down, __uint_as_float(raw[i] & 0xFFFF0000u) * down);
        qsc[nt][0] = __shfl_sync(0xffffffffu, up, 8 * c);
        qsc[nt][1] = __shfl_sync(0xffffffffu, up, 8 * c + 4);
      } else {
#pragma unroll
        for (int i = 0; i < QW; ++i) qf[nt][i] = raw[i];
        qsc[nt][0] = qsc[nt][1] = 1.f;
      }
    }
    // ---- phase 1: scores of the chunk, s[h][key] = q_h . k_key
    bool ok = true;
    for (int tl = 0; tl < wk.ntl; ++tl, ++it) {
      const int s = it % STAGES;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_full(s), (it / STAGES) & 1, abort_flag, err));
      if (!ok) continue;
      const uint8_t* tile = smem + s * TILE_BYTES;
      // K rows 16 warp + g and + 8: this thread's slice [c DQ, (c+1) DQ) of each
      uint32_t ka[2][KW];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = 16 * kblk + g + 8 * r;
#pragma unroll
        for (int j = 0; j < KW / 4; ++j) {
          const uint4 u = *reinterpret_cast<const uint4*>(tile + tile_off<HD, KV8>(row, c * DQ * GE::ESZ + 16 * (j ^ rot)));
          ka[r][4 * j + 0] = u.x;
          ka[r][4 * j + 1] = u.y;
          ka[r][4 * j + 2] = u.z;
          ka[r][4 * j + 3] = u.w;
        }
      }
      // two partial sums per column block (even and odd K steps): twice the independent
      // MMAs in flight against the MMA latency
      float acc[NTW][4], acc2[NTW][4];
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = acc2[nt][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
        // MMA K index 2c + {0, 1} -> d = c DQ + 4 kk + {0, 1}; 2c + 8 + {0, 1} -> + {2, 3}
        uint32_t a0, a1, a2, a3;
        if constexpr (KV8) {
          a0 = e4m3x2_f16x2<false>(ka[0][kk]);
          a1 = e4m3x2_f16x2<false>(ka[1][kk]);
          a2 = e4m3x2_f16x2<true>(ka[0][kk]);
          a3 = e4m3x2_f16x2<true>(ka[1][kk]);
        } else {
          a0 = ka[0][2 * kk];
          a1 = ka[1][2 * kk];
          a2 = ka[0][2 * kk + 1];
          a3 = ka[1][2 * kk + 1];
        }
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
          mma16816<KV8>((kk & 1) ? acc2[nt] : acc[nt], a0, a1, a2, a3, qf[nt][2 * kk], qf[nt][2 * kk + 1]);
      }
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
      // the MMAs above have consumed every value this warp read from the slot
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty(s));
      // acc[nt] = S^T: rows keys 16 kblk + g (+8), columns heads 8 (nt0 + nt) + 2c (+1)
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 8 * (nt0 + nt) + 2 * c + (e & 1);
          const int key = tl * TILE + 16 * kblk + g + 8 * (e >> 1);
          if (h < G) work[h * wstride + key] = key < wk.n_valid ? acc[nt][e] * qsc[nt][e & 1] : -CUDART_INF_F;
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
    // ---- phase 2: chunk softmax per head (exp2 domain), p written in place
    const int nk_pad = wk.ntl * TILE;
    for (int h = warp; h < G; h += NCW) {
      float* sh = work + h * wstride;
      float mx = -CUDART_INF_F;
      for (int j = lane; j < nk_pad; j += 32) mx = fmaxf(mx, sh[j]);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m = (mx == -CUDART_INF_F) ? 0.f : mx * c_log2;
      float sum = 0.f;
      // p in the P V operand type (f16 for fp8 caches, else bf16), written in place over the
      // scores: p_j lands in the bytes of score j / 2, which the warp has already read (in an
      // earlier pass, or, for j < 32, by the load of this pass)
      const uint32_t sh16 = smem_u32(sh);
      for (int j = lane; j < nk_pad; j += 32) {
        const float pv = ex2_approx(fmaf(sh[j], c_log2, -m));
        st_shared_u16(sh16 + 2 * j, KV8 ? __half_as_ushort(__float2half_rn(pv))
                                        : __bfloat16_as_ushort(__float2bfloat16_rn(pv)));
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
    // ---- phase 3: O^T = V^T P^T for head-dimension rows [16 MT mblk, +16 MT) and column
    // blocks [pt0, pt0 + NTP)
    float oacc[MT][NTP][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NTP; ++nt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
    const int dbase = mblk * 16 * MT + DV * g;   // this thread's head-dimension elements dbase .. + DV - 1
    for (int tl = 0; tl < wk.ntl; ++tl, ++it) {
      const int s = it % STAGES;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_full(s), (it / STAGES) & 1, abort_flag, err));
      if (!ok) continue;
      const uint8_t* tile = smem + s * TILE_BYTES;
      const int valid_here = wk.n_valid - tl * TILE;   // keys of this tile inside the sequence
      // a full tile takes the copy of the loop without the per-key check (only a chunk's
      // last tile can reach past the sequence)
      auto tile_pv = [&](auto mask_tag) {
      constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
      for (int ks = 0; ks < TILE / 16; ++ks) {
        // the MMA K index 2c + {0, 1, 8, 9} is key 16 ks + 2c + {0, 1, 8, 9}
        uint32_t vw[4][DV * GE::ESZ / 4 > 0 ? DV * GE::ESZ / 4 : 1];   // V[key][dbase .. + DV) per key
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = 16 * ks + 2 * c + (i & 1) + 8 * (i >> 1);
          const uint32_t off = tile_off<HD, KV8>(key, dbase * GE::ESZ);
          const bool in = !MASK || key < valid_here;
          if constexpr (DV * GE::ESZ == 8) {
            const uint2 u = *reinterpret_cast<const uint2*>(tile + off);
            vw[i][0] = in ? u.x : 0u;
            vw[i][1] = in ? u.y : 0u;
          } else if constexpr (DV * GE::ESZ == 4) {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(tile + off);
            vw[i][0] = in ? u : 0u;
          } else {   // fp8, D = 64: two codes
            const uint32_t u = *reinterpret_cast<const uint16_t*>(tile + off);
            vw[i][0] = in ? u : 0u;
          }
        }
        // A fragments: block mt covers d = dbase + 2 mt (MMA row g) and + 1 (row g + 8)
        uint32_t af[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int pr = 0; pr < 2; ++pr) {   // pr 0: keys (2c, 2c+1); pr 1: keys (2c+8, 2c+9)
            const int i0 = 2 * pr, i1 = 2 * pr + 1;
            uint32_t lo, hi;   // (key i0, key i1) at d = dbase + 2mt, and at + 1
            if constexpr (KV8) {
              const uint32_t x = prmt(vw[i0][0], vw[i1][0], mt == 0 ? 0x5140u : 0x7362u);
              lo = e4m3x2_f16x2<false>(x);
              hi = e4m3x2_f16x2<true>(x);
            } else {
              lo = prmt(vw[i0][mt], vw[i1][mt], 0x5410u);
              hi = prmt(vw[i0][mt], vw[i1][mt], 0x7632u);
            }
            af[mt][2 * pr + 0] = lo;
            af[mt][2 * pr + 1] = hi;
          }
        }
        // B fragments: P^T, keys (2c, 2c+1) and (2c+8, 2c+9) of head 8 (pt0 + nt) + g
#pragma unroll
        for (int nt = 0; nt < NTP; ++nt) {
          const int h = 8 * (pt0 + nt) + g;
          uint32_t b0 = 0u, b1 = 0u;
          if (h < G) {   // p of keys (2c, 2c+1) and (2c+8, 2c+9), already in the operand type
            const uint16_t* ph = reinterpret_cast<const uint16_t*>(work + h * wstride) + tl * TILE + 16 * ks + 2 * c;
            b0 = *reinterpret_cast<const uint32_t*>(ph);
            b1 = *reinterpret_cast<const uint32_t*>(ph + 8);
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            mma16816<KV8>(oacc[mt][nt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
        }
      }
      };
      if (valid_here >= TILE) tile_pv(std::false_type{});
      else tile_pv(std::true_type{});
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty(s));
    }
    // ---- write the chunk's O_c (normalised, times v_scale) and LSE_c
    {
      const size_t base = (static_cast<size_t>(wk.b) * Hq + h0) * S_max + wk.c;
#pragma unroll
      for (int nt = 0; nt < NTP; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 8 * (pt0 + nt) + 2 * c + e;
          if (h >= G) continue;
          const float sc = v_scale / st_l[h];
          float* dst = ws_o + (base + static_cast<size_t>(h) * S_max) * HD + dbase;
          if constexpr (DV == 4) {
            // elements dbase + {0, 1, 2, 3} = (mt 0 row g, mt 0 row g+8, mt 1 row g, mt 1 row g+8)
            st_global_hint(dst, oacc[0][nt][e] * sc, oacc[0][nt][2 + e] * sc, oacc[MT - 1][nt][e] * sc,
                           oacc[MT - 1][nt][2 + e] * sc, keep_policy);
          } else {
            st_global_hint(dst, oacc[0][nt][e] * sc, oacc[0][nt][2 + e] * sc, keep_policy);
          }
        }
      }
      if (tid < G)
        st_global_hint(ws_lse + base + static_cast<size_t>(tid) * S_max,
                       (st_m[tid] + log2f(st_l[tid])) * 0.69314718055994531f, keep_policy);
      if (tid == 0) *stop = *abort_flag;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");  // scores and stats free for the next item
    if (*stop) break;
  }
}

}  // namespace decode_mma

// One CTA per (b, h): LSE-weighted merge of the chunk results.  The four warps
// take chunks w, w + 4, w + 8, ... and issue up to 16 chunk loads (lane l:
// head-dimension elements [l HD/32, (l+1) HD/32)) before any arithmetic, so a
// sequence of up to 64 chunks is read in one round of memory latency; each warp
// keeps a running (max, sum, weighted O) over its chunks, and warp 0 merges the
// four through shared memory.  (One warp walking all chunks of its (b, h) made
// the longest sequences' warps wait for one round per 8-16 chunks.)
template <int HDIM>
__global__ void __launch_bounds__(128)
attn_decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                           const int* __restrict__ seqlens, __nv_bfloat16* __restrict__ o,
                           float* __restrict__ lse, int B, int Hq, int Nk_max, int chunk, int S_max,
                           int* err) {
  constexpr int E = HDIM / 32;   // elements per lane: 4 or 2
  constexpr int NW = 4;          // warps
  constexpr int DEPTH = 16;      // chunks per warp per round
  constexpr float LOG2E = 1.4426950408889634f;
  __shared__ float s_m[NW], s_s[NW];
  __shared__ __align__(16) float s_acc[NW][HDIM];
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());
  const int bh = static_cast<int>(blockIdx.x);
  const int b = bh / Hq;
  const int Lb = __ldg(seqlens + b);
  __nv_bfloat16* orow = o + static_cast<size_t>(bh) * HDIM + lane * E;
  if (Lb < 1 || Lb > Nk_max) {   // the whole CTA leaves together
    if (warp == 0) {
      if (lane == 0) atomicCAS(err, 0, ATTN_ERR_SEQLEN);
      if constexpr (E == 4) *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
      else *reinterpret_cast<uint32_t*>(orow) = 0u;
      if (lane == 0 && lse != nullptr) lse[bh] = -CUDART_INF_F;
    }
    return;
  }
  const int n = (Lb + chunk - 1) / chunk;
  const float* lp = ws_lse + static_cast<size_t>(bh) * S_max;
  const float* op = ws_o + static_cast<size_t>(bh) * S_max * HDIM + lane * E;
  float m = -CUDART_INF_F, s = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int c0 = warp; c0 < n; c0 += NW * DEPTH) {   // c0 < n: lv[0] is finite
    float lv[DEPTH];
    float x[DEPTH][E];
#pragma unroll
    for (int u = 0; u < DEPTH; ++u) {
      // chunks past n re-read chunk n - 1 (no branch, so every load can issue at once)
      // and get LSE -inf, i.e. weight 0
      // (volatile asm loads keep the compiler from spreading them over several rounds)
      const int c = c0 + NW * u;
      const int cc = min(c, n - 1);
      float l;
      asm volatile("ld.global.f32 %0, [%1];" : "=f"(l) : "l"(lp + cc));
      lv[u] = c < n ? l : -CUDART_INF_F;
      const float* src = op + static_cast<size_t>(cc) * HDIM;
      if constexpr (E == 4)
        asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(x[u][0]), "=f"(x[u][1]), "=f"(x[u][2]), "=f"(x[u][3]) : "l"(src));
      else
        asm volatile("ld.global.v2.f32 {%0, %1}, [%2];" : "=f"(x[u][0]), "=f"(x[u][1]) : "l"(src));
    }
    float mr = lv[0];
#pragma unroll
    for (int u = 1; u < DEPTH; ++u) mr = fmaxf(mr, lv[u]);
    const float mn = fmaxf(m, mr);
    const float corr = ex2_approx((m - mn) * LOG2E);   // 0 on the first round (m = -inf)
    s *= corr;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= corr;
#pragma unroll
    for (int u = 0; u < DEPTH; ++u) {
      const float w = ex2_approx((lv[u] - mn) * LOG2E);
      s += w;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(w, x[u][e], acc[e]);
    }
    m = mn;
  }
  // warps without chunks (n < 4) keep m = -inf, s = 0, acc = 0
  if (lane == 0) {
    s_m[warp] = m;
    s_s[warp] = s;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc[e];
  __syncthreads();
  if (warp != 0) return;
  float M = s_m[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) M = fmaxf(M, s_m[w]);
  float S = 0.f;
  float out[E];
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const float f = s_m[w] == -CUDART_INF_F ? 0.f : ex2_approx((s_m[w] - M) * LOG2E);
    S = fmaf(f, s_s[w], S);
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = fmaf(f, s_acc[w][lane * E + e], out[e]);
  }
  const float inv = 1.f / S;
  if constexpr (E == 4)
    *reinterpret_cast<uint2*>(orow) =
        make_uint2(pack_bf16x2(out[0] * inv, out[1] * inv), pack_bf16x2(out[2] * inv, out[3] * inv));
  else
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(out[0] * inv, out[1] * inv);
  if (lane == 0 && lse != nullptr) lse[bh] = M + logf(S);
}

template <int G, bool PAGED>
int launch_split(const CUtensorMap& tk, const CUtensorMap& tv, const void* q, const int* seqlens,
                 float* ws_o, float* ws_lse, int B, int Hq, int Hkv, int Nk_max, float scale,
                 int chunk, int S_max, int num_sms, cudaStream_t stream, int* err, const Paging& pg,
                 float k_scale, float v_scale) {
  const Layout L = layout(G, chunk, B, Ring<G>::RING_BYTES);
  const int smem = L.bytes + 1024;
  // the persistent grid is as many CTAs as are resident at once: up to three
  // per SM, fewer when a large chunk or head group enlarges the score area
  static KernelSetup setup;
  int n = 0;
  if (const int rc = prepare_kernel(setup, attn_decode_splitkv_kernel<G, PAGED>, smem, NTHREADS, &n);
      rc != ATTN_OK)
    return rc;
  constexpr int cap = Ring<G>::CTAS_PER_SM;
  const int resident = n < 1 ? 1 : (n > cap ? cap : n);
  const int grid = resident * num_sms;
  attn_decode_splitkv_kernel<G, PAGED><<<grid, NTHREADS, smem, stream>>>(
      tk, tv, static_cast<const __nv_bfloat16*>(q), seqlens, ws_o, ws_lse, B, Hq, Hkv, Nk_max, chunk,
      S_max, scale * 1.4426950408889634f, err, pg);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int HDIM, int G, bool PAGED, bool KV8>
int launch_mma(const CUtensorMap& tk, const CUtensorMap& tv, const void* q, const int* seqlens, float* ws_o,
               float* ws_lse, int B, int Hq, int Hkv, int Nk_max, float scale, int chunk, int S_max,
               int num_sms, cudaStream_t stream, int* err, const Paging& pg, float k_scale, float v_scale) {
  using C = decode_mma::Cfg<HDIM, G, KV8>;
  constexpr int tile = decode_mma::Geo<HDIM, KV8>::TILE_BYTES;
  constexpr int kMaxSmem = 227 * 1024;
  int stages = C::SMALL_RING_BYTES / tile;
  if (G > 8) {
    // as many ring slots as fit next to the scores with two CTAs per SM, else with one
    // (long chunks), at most MAX_STAGES
    const int rest = decode_mma::layout(G, chunk, B, 0).bytes + 1024;
    stages = (kMaxSmem / 2 - 1024 - rest) / tile;
    if (stages < 2) stages = (kMaxSmem - rest) / tile;
    if (stages > decode_mma::MAX_STAGES) stages = decode_mma::MAX_STAGES;
  }
  if (stages < 2) return ATTN_ERR_CAPACITY;
  const decode_mma::Layout L = decode_mma::layout(G, chunk, B, stages * tile);
  const int smem = L.bytes + 1024;
  if (smem > kMaxSmem) return ATTN_ERR_CAPACITY;
  static KernelSetup setup;
  int n = 0;
  if (const int rc = prepare_kernel(setup, decode_mma::attn_decode_mma_kernel<HDIM, G, PAGED, KV8>, smem,
                                    C::NTHREADS, &n);
      rc != ATTN_OK)
    return rc;
  const int resident = n < 1 ? 1 : (n > C::CTAS_PER_SM ? C::CTAS_PER_SM : n);
  decode_mma::attn_decode_mma_kernel<HDIM, G, PAGED, KV8><<<resident * num_sms, C::NTHREADS, smem, stream>>>(
      tk, tv, static_cast<const __nv_bfloat16*>(q), seqlens, ws_o, ws_lse, B, Hq, Hkv, Nk_max, chunk, S_max,
      scale * k_scale * 1.4426950408889634f, v_scale, err, pg, stages);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Tensor maps over a contiguous cache [B, Nk_max, Hkv, D] or a page pool
// [num_pages, page_size, Hkv, D].  SIMT kernel: one box is 64 key rows of one
// KV head, unswizzled.  Tensor-core kernel: one box is one swizzled slab (64
// key rows x at most 128 bytes of one KV head).
inline bool cache_maps(CUtensorMap* tk, CUtensorMap* tv, const void* k, const void* v, int D, int Hkv,
                       int rows, int outer, bool kv8, bool mma) {
  const CUtensorMapDataType dt = kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t es = kv8 ? 1 : 2;
  uint32_t box[4] = {static_cast<uint32_t>(D), 1, TILE, 1};
  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (mma) {
    const uint32_t row = static_cast<uint32_t>(D) * es;
    const uint32_t srow = row > 128 ? 128 : row;
    box[0] = srow / es;
    swz = srow == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  }
  return encode_tiled_4d(tk, dt, k, D, Hkv, rows, outer, es, box, swz) &&
         encode_tiled_4d(tv, dt, v, D, Hkv, rows, outer, es, box, swz);
}

// The SIMT kernel serves the bf16 cache with D = 128 and up to 8 query heads
// per KV head (it keeps up with HBM there); every other case takes the
// tensor-core kernel.
inline bool use_simt(int D, int G, bool kv8) { return !kv8 && D == 128 && G <= 8; }

template <bool PAGED, bool KV8>
int launch_split_any(const void* k, const void* v, int map_rows, int map_outer, const void* q,
                     const int* seqlens, void* workspace, int B, int Hq, int Hkv, int Nk_max, int D,
                     float scale, int chunk, int num_sms, cudaStream_t stream, int* err, const Paging& pg,
                     float k_scale, float v_scale) {
  const int S_max = (Nk_max + chunk - 1) / chunk;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_lse = ws_o + static_cast<size_t>(B) * Hq * S_max * D;
  const int G = Hq / Hkv;
  const bool simt = use_simt(D, G, KV8);
  CUtensorMap tk, tv;
  if (!cache_maps(&tk, &tv, k, v, D, Hkv, map_rows, map_outer, KV8, !simt)) return ATTN_ERR_CUDA;
#define ATTN_SPLIT_ARGS tk, tv, q, seqlens, ws_o, ws_lse, B, Hq, Hkv, Nk_max, scale, chunk, S_max, \
                        num_sms, stream, err, pg, k_scale, v_scale
  if (simt) {
    if constexpr (!KV8) {
      switch (G) {
        case 1: return launch_split<1, PAGED>(ATTN_SPLIT_ARGS);
        case 2: return launch_split<2, PAGED>(ATTN_SPLIT_ARGS);
        case 4: return launch_split<4, PAGED>(ATTN_SPLIT_ARGS);
        case 8: return launch_split<8, PAGED>(ATTN_SPLIT_ARGS);
        default: return ATTN_ERR_GQA;
      }
    }
    return ATTN_ERR_GQA;
  }
  if (D == 128) {
    switch (G) {
      case 1: return launch_mma<128, 1, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 2: return launch_mma<128, 2, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 4: return launch_mma<128, 4, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 8: return launch_mma<128, 8, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 16: return launch_mma<128, 16, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 32: return launch_mma<128, 32, PAGED, KV8>(ATTN_SPLIT_ARGS);
      default: return ATTN_ERR_GQA;
    }
  }
  if (D == 64) {
    switch (G) {
      case 1: return launch_mma<64, 1, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 2: return launch_mma<64, 2, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 4: return launch_mma<64, 4, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 8: return launch_mma<64, 8, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 16: return launch_mma<64, 16, PAGED, KV8>(ATTN_SPLIT_ARGS);
      case 32: return launch_mma<64, 32, PAGED, KV8>(ATTN_SPLIT_ARGS);
      default: return ATTN_ERR_GQA;
    }
  }
#undef ATTN_SPLIT_ARGS
  return ATTN_ERR_HEAD_DIM;
}

}  // namespace decode

int launch_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                          const int* seqlens, void* workspace, int B, int Hq, int Hkv,
                          int Nk_max, int D, float scale, int chunk, int num_sms, cudaStream_t stream,
                          int* err, int kv8, float k_scale, float v_scale) {
  using namespace decode;
  const Paging none{nullptr, 0, 0, 0};
  return kv8 ? launch_split_any<false, true>(k_cache, v_cache, Nk_max, B, q, seqlens, workspace, B, Hq, Hkv,
                                             Nk_max, D, scale, chunk, num_sms, stream, err, none, k_scale, v_scale)
             : launch_split_any<false, false>(k_cache, v_cache, Nk_max, B, q, seqlens, workspace, B, Hq, Hkv,
                                              Nk_max, D, scale, chunk, num_sms, stream, err, none, 1.f, 1.f);
}

int launch_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int* block_table, const int* seqlens, void* workspace, int B,
                                int Hq, int Hkv, int num_pages, int page_size, int max_pages, int D,
                                float scale, int chunk, int num_sms, cudaStream_t stream, int* err,
                                int kv8, float k_scale, float v_scale) {
  using namespace decode;
  const Paging pg{block_table, max_pages, page_size, num_pages};
  return kv8 ? launch_split_any<true, true>(k_pages, v_pages, page_size, num_pages, q, seqlens, workspace, B,
                                            Hq, Hkv, max_pages * page_size, D, scale, chunk, num_sms, stream,
                                            err, pg, k_scale, v_scale)
             : launch_split_any<true, false>(k_pages, v_pages, page_size, num_pages, q, seqlens, workspace, B,
                                             Hq, Hkv, max_pages * page_size, D, scale, chunk, num_sms, stream,
                                             err, pg, 1.f, 1.f);
}

int launch_decode_combine(const void* workspace, const int* seqlens, void* o, float* lse, int B,
                          int Hq, int Nk_max, int D, int chunk, cudaStream_t stream, int* err) {
  using namespace decode;
  const int S_max = (Nk_max + chunk - 1) / chunk;
  const float* ws_o = static_cast<const float*>(workspace);
  const float* ws_lse = ws_o + static_cast<size_t>(B) * Hq * S_max * D;
  const int grid = B * Hq;
  if (D == 128)
    attn_decode_combine_kernel<128><<<grid, 128, 0, stream>>>(ws_o, ws_lse, seqlens, static_cast<__nv_bfloat16*>(o),
                                                              lse, B, Hq, Nk_max, chunk, S_max, err);
  else if (D == 64)
    attn_decode_combine_kernel<64><<<grid, 128, 0, stream>>>(ws_o, ws_lse, seqlens, static_cast<__nv_bfloat16*>(o),
                                                             lse, B, Hq, Nk_max, chunk, S_max, err);
  else
    return ATTN_ERR_HEAD_DIM;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

// kernels.h — launchers shared between the C-ABI translation unit and the
// kernel translation units.  Arguments are validated by the caller (attn_abi.cu).
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn.h"

namespace attn {

constexpr int kMaxDevices = 64;

// Per-device launch set-up of one kernel: the dynamic shared-memory limit it
// was raised to and the CTAs per SM resident at the last size asked for.
// One object per kernel instance (a function-local static); every access holds
// its mutex, so concurrent callers on any devices are safe.
struct KernelSetup {
  std::mutex mu;
  int smem_limit[kMaxDevices] = {};   // 0: attribute not raised on that device yet
  int occ_smem[kMaxDevices] = {};     // shared-memory size resident[] was computed for
  int resident[kMaxDevices] = {};
};

// Raises `kernel`'s dynamic shared-memory limit on the current device to at
// least `smem` bytes (once per device) and, when `resident` is given, stores
// the number of CTAs of `threads` threads and `smem` bytes that fit on one SM.
template <typename Kernel>
int prepare_kernel(KernelSetup& st, Kernel kernel, int smem, int threads = 0, int* resident = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(st.mu);
  if (st.smem_limit[dev] < smem) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    st.smem_limit[dev] = smem;
  }
  if (resident != nullptr) {
    if (st.occ_smem[dev] != smem) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess)
        return ATTN_ERR_CUDA;
      st.resident[dev] = n;
      st.occ_smem[dev] = smem;
    }
    *resident = st.resident[dev];
  }
  return ATTN_OK;
}

struct FwdParams {
  void* o;           // bf16 or fp16 output
  float* lse;
  int B, Hq, Hkv, Nq, Nk;
  int group;         // Hq / Hkv
  float scale_log2;  // scale * log2(e)
  int causal, window;
  int* err;          // device error word
  // ragged batches: Q/O [total_q, Hq, D], K/V [total_k, Hkv, D]; sequence b owns
  // rows cu_q[b] .. cu_q[b+1]-1 (queries) and cu_k[b] .. cu_k[b+1]-1 (keys); Nq is
  // then the maximum query length (it sizes the unit list)
  int varlen;
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
  // softcap c > 0: score s -> c * tanh(scale * s / c); cap_pre = scale / c,
  // cap_post = c * log2(e).  sinks: one logit per query head (natural-log
  // units) in every row's softmax denominator, or null.
  float cap_pre, cap_post;
  // Softcap fast paths: on a tile whose raw scores all satisfy |s| <= cap_smax_short
  // (cap_smax_long) the capped score in exp2 units is s * P(s^2) with
  // P(w) = sum_k cap_short[k] w^k (cap_long[k] w^k): tanh as an odd minimax
  // polynomial.  A negative bound disables that path.
  float cap_short[4];
  float cap_long[6];
  float cap_smax_short, cap_smax_long;
  const float* sinks;
  float o_scale;     // multiplies O (the V dequantisation scale of E4M3 inputs; else 1)
  int o_align32;     // O is 32-byte aligned (rows are then written with 32-byte stores)
};

// Tensor maps (cuTensorMapEncodeTiled, fetched from the driver at run time).
// Dimensions are innermost first; strides are packed (contiguous tensor).
bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t d0,
                     uint64_t d1, uint64_t d2, uint32_t esize, const uint32_t box[3],
                     CUtensorMapSwizzle swz);
bool encode_tiled_4d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t d0,
                     uint64_t d1, uint64_t d2, uint64_t d3, uint32_t esize, const uint32_t box[4],
                     CUtensorMapSwizzle swz);

// Tensor-core forward; f16 != 0 selects fp16 operands and output instead of bf16.
// With cu_q != nullptr the batch is ragged (packed token-major layout, see FwdParams);
// Nq is then the maximum query length and Nk is unused.
// softcap > 0 (bf16 only) caps the scaled scores; sinks (device, [Hq]) adds
// one logit per query head to every row's softmax denominator.
int launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, int f16, float scale, int causal, int window,
                  int num_sms, cudaStream_t stream, int* err, const int* cu_q = nullptr,
                  const int* cu_k = nullptr, int total_q = 0, int total_k = 0,
                  float softcap = 0.f, const float* sinks = nullptr);

// Backward: D and LSE*log2(e) into the workspace (bwd_workspace_bytes), dQ
// zeroed and accumulated in fp32, dK and dV written in bf16.  Head dimension
// D = 64 or 128.
size_t bwd_workspace_bytes(int B, int Hq, int Nq);
// fp8 prefill: E4M3 q [B,Hq,Nq,128], k / v [B,Hkv,Nk,128] (codes, per-tensor
// scales); V is widened to bf16 into `workspace` (fwd_fp8_workspace_bytes) first.
size_t fwd_fp8_workspace_bytes(int B, int Hkv, int Nk, int D);
int launch_fwd_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                   float v_scale, void* o, float* lse, void* workspace, int B, int Hq, int Hkv,
                   int Nq, int Nk, int D, float scale, int causal, int window, int num_sms,
                   cudaStream_t stream, int* err);
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
               const float* lse, float* dq, void* dk, void* dv, void* workspace, int B, int Hq,
               int Hkv, int Nq, int Nk, int D, float scale, int causal, int window, cudaStream_t stream,
               int* err);

int launch_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                    int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
                    cudaStream_t stream, int* err);

// Split-KV decode, partial step.  kv8 != 0: the cache holds fp8 E4M3 codes
// whose values are code * k_scale (K) and code * v_scale (V); else bf16
// (k_scale, v_scale unused).
int launch_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                          const int* seqlens, void* workspace, int B, int Hq, int Hkv,
                          int Nk_max, int D, float scale, int chunk, int num_sms, cudaStream_t stream,
                          int* err, int kv8 = 0, float k_scale = 1.f, float v_scale = 1.f);

int launch_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int* block_table, const int* seqlens, void* workspace, int B,
                                int Hq, int Hkv, int num_pages, int page_size, int max_pages, int D,
                                float scale, int chunk, int num_sms, cudaStream_t stream, int* err,
                                int kv8 = 0, float k_scale = 1.f, float v_scale = 1.f);

int launch_decode_combine(const void* workspace, const int* seqlens, void* o, float* lse, int B,
                          int Hq, int Nk_max, int D, int chunk, cudaStream_t stream, int* err);

}  // namespace attn

// attn_abi.cu — the C ABI declared in include/attn.h: argument validation,
// device checks, the device error word and tensor-map encoding.
//
// Host-side validation runs before any CUDA call, so argument errors are
// reported without touching a GPU.  Nothing here allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn.h"
#include "kernels.h"

namespace attn {

// Per-device error word written by kernels (bounded-wait timeouts, bad
// sequence lengths) and read / cleared by attn_get_device_error().
__device__ int g_device_error;

namespace {

struct DeviceInfo {
  bool ready = false;
  int status = ATTN_OK;
  int* err = nullptr;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device: must be compute capability 10.3.  Fills the error-word
// address and SM count once per device.
int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (major != 10 || minor != 3) {
      d.status = ATTN_ERR_DEVICE;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return ATTN_ERR_CUDA;
      d.err = static_cast<int*>(p);
      d.status = ATTN_OK;
    }
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  if (d.status != ATTN_OK) return d.status;
  *out = &d;
  return ATTN_OK;
}

int check_common(const void* q, const void* k, const void* v, const void* o, const void* lse,
                 int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale) {
  if (!q || !k || !v || !o) return ATTN_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || D <= 0) return ATTN_ERR_DIM;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_DIM;  // fp32 grid y / z limits
  if (Hq % Hkv != 0) return ATTN_ERR_GQA;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
    return ATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  return ATTN_OK;
}

}  // namespace

bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t d0,
                     uint64_t d1, uint64_t d2, uint32_t esize, const uint32_t box[3],
                     CUtensorMapSwizzle swz) {
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_4d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t d0,
                     uint64_t d1, uint64_t d2, uint64_t d3, uint32_t esize, const uint32_t box[4],
                     CUtensorMapSwizzle swz) {
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * esize, d0 * d1 * esize, d0 * d1 * d2 * esize};
  const cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return g_encode(map, dt, 4, const_cast<void*>(base), dims, strides, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace attn

using namespace attn;

extern "C" {

static int fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, int f16, float scale, int causal, int window,
                  attn_stream_t stream) {
  int rc = check_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale);
  if (rc != ATTN_OK) return rc;
  if (D != 64 && D != 128) return ATTN_ERR_HEAD_DIM;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return launch_fwd_tc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, f16, scale, causal, window,
                       dev->num_sms, reinterpret_cast<cudaStream_t>(stream), dev->err);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
             attn_stream_t stream) {
  return fwd_tc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, 0, scale, causal, window, stream);
}
int attn_fwd_softcap_sink(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                          int window, float softcap, const float* sinks, attn_stream_t stream) {
  int rc = check_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale);
  if (rc != ATTN_OK) return rc;
  if (D != 64 && D != 128) return ATTN_ERR_HEAD_DIM;
  if (!std::isfinite(softcap)) return ATTN_ERR_SCALE;
  if (sinks != nullptr && (reinterpret_cast<uintptr_t>(sinks) & 3u) != 0) return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return launch_fwd_tc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, 0, scale, causal, window,
                       dev->num_sms, reinterpret_cast<cudaStream_t>(stream), dev->err, nullptr,
                       nullptr, 0, 0, softcap, sinks);
}

int attn_fwd_fp16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
                  attn_stream_t stream) {
  return fwd_tc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, 1, scale, causal, window, stream);
}

size_t attn_fwd_fp8_workspace_size(int B, int Hkv, int Nk, int D) {
  if (B <= 0 || Hkv <= 0 || Nk <= 0 || D <= 0) return 0;
  return fwd_fp8_workspace_bytes(B, Hkv, Nk, D);
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                 float v_scale, void* o, float* lse, void* workspace, int B, int Hq, int Hkv,
                 int Nq, int Nk, int D, float scale, int causal, int window, attn_stream_t stream) {
  int rc = check_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale);
  if (rc != ATTN_OK) return rc;
  if (!workspace) return ATTN_ERR_NULL;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  if (D != 128) return ATTN_ERR_HEAD_DIM;
  for (const float x : {q_scale, k_scale, v_scale})
    if (!std::isfinite(x) || !(x > 0.f)) return ATTN_ERR_SCALE;
  const float s_all = scale * q_scale * k_scale;  // the score scale the kernel applies
  if (!std::isfinite(s_all) || !(s_all > 0.f)) return ATTN_ERR_SCALE;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return launch_fwd_fp8(q, k, v, q_scale, k_scale, v_scale, o, lse, workspace, B, Hq, Hkv, Nq, Nk,
                        D, scale, causal, window, dev->num_sms,
                        reinterpret_cast<cudaStream_t>(stream), dev->err);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq, int Hkv,
                    int max_seqlen_q, int total_q, int total_k, int D, float scale, int causal,
                    int window, attn_stream_t stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return ATTN_ERR_NULL;
  int rc = check_common(q, k, v, o, lse, B, Hq, Hkv, max_seqlen_q, total_k, D, scale);
  if (rc != ATTN_OK) return rc;
  if (total_q <= 0) return ATTN_ERR_DIM;
  if (!aligned16(cu_seqlens_q) || !aligned16(cu_seqlens_k)) return ATTN_ERR_ALIGN;
  if (D != 64 && D != 128) return ATTN_ERR_HEAD_DIM;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return launch_fwd_tc(q, k, v, o, lse, B, Hq, Hkv, max_seqlen_q, 0, D, 0, scale, causal, window,
                       dev->num_sms, reinterpret_cast<cudaStream_t>(stream), dev->err,
                       cu_seqlens_q, cu_seqlens_k, total_q, total_k);
}

int attn_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                  int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
                  attn_stream_t stream) {
  int rc = check_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale);
  if (rc != ATTN_OK) return rc;
  if (D != 32 && D != 64 && D != 128) return ATTN_ERR_HEAD_DIM;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return (launch_fwd_fp32(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window,
                                reinterpret_cast<cudaStream_t>(stream), dev->err));
}

size_t attn_decode_workspace_size(int B, int Hq, int D, int Nk_max, int chunk) {
  if (B <= 0 || Hq <= 0 || D <= 0 || Nk_max <= 0 || chunk <= 0) return 0;
  const size_t S_max = (static_cast<size_t>(Nk_max) + chunk - 1) / chunk;
  const size_t rows = static_cast<size_t>(B) * Hq * S_max;
  const size_t bytes = rows * (static_cast<size_t>(D) + 1) * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

static int check_decode(int B, int Hq, int Hkv, int Nk_max, int D, int chunk) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nk_max <= 0 || D <= 0 || chunk <= 0) return ATTN_ERR_DIM;
  if (Hq % Hkv != 0) return ATTN_ERR_GQA;
  const int g = Hq / Hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16 && g != 32) return ATTN_ERR_GQA;
  if (D != 64 && D != 128) return ATTN_ERR_HEAD_DIM;
  if (chunk % 64 != 0 || chunk > 1024) return ATTN_ERR_CHUNK;
  if (B > 4096) return ATTN_ERR_CAPACITY;
  if (static_cast<long long>(B) * Hq > (1ll << 30)) return ATTN_ERR_DIM;
  return ATTN_OK;
}

int attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                        const int* seqlens, void* workspace, int B, int Hq, int Hkv, int Nk_max,
                        int D, float scale, int chunk, attn_stream_t stream) {
  if (!q || !k_cache || !v_cache || !seqlens || !workspace) return ATTN_ERR_NULL;
  int rc = check_decode(B, Hq, Hkv, Nk_max, D, chunk);
  if (rc != ATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace) ||
      !aligned16(seqlens))
    return ATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return (launch_decode_splitkv(q, k_cache, v_cache, seqlens, workspace, B, Hq, Hkv, Nk_max, D,
                                      scale, chunk, dev->num_sms,
                                      reinterpret_cast<cudaStream_t>(stream), dev->err));
}

int attn_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int* block_table, const int* seqlens, void* workspace, int B,
                              int Hq, int Hkv, int num_pages, int page_size, int max_pages, int D,
                              float scale, int chunk, attn_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !seqlens || !workspace) return ATTN_ERR_NULL;
  if (num_pages <= 0 || max_pages <= 0 || page_size <= 0 || page_size % 64 != 0) return ATTN_ERR_DIM;
  if (static_cast<long long>(max_pages) * page_size > 0x7fffffffLL) return ATTN_ERR_DIM;
  int rc = check_decode(B, Hq, Hkv, max_pages * page_size, D, chunk);
  if (rc != ATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(workspace) ||
      !aligned16(seqlens) || !aligned16(block_table))
    return ATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return launch_decode_splitkv_paged(q, k_pages, v_pages, block_table, seqlens, workspace, B, Hq,
                                     Hkv, num_pages, page_size, max_pages, D, scale, chunk,
                                     dev->num_sms, reinterpret_cast<cudaStream_t>(stream), dev->err);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Nq) {
  if (B <= 0 || Hq <= 0 || Nq <= 0) return 0;
  return bwd_workspace_bytes(B, Hq, Nq);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, float* dq, void* dk, void* dv, void* workspace, int B, int Hq,
             int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
             attn_stream_t stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_ERR_NULL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || D <= 0) return ATTN_ERR_DIM;
  if (Hq % Hkv != 0) return ATTN_ERR_GQA;
  if (D != 64 && D != 128) return ATTN_ERR_HEAD_DIM;
  if (static_cast<long long>(B) * Hq * Nq > (1ll << 31) || static_cast<long long>(B) * Hkv > 65535 ||
      B > 65535)
    return ATTN_ERR_DIM;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return ATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != ATTN_OK) return rc;
  return launch_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, Hq, Hkv, Nq, Nk, D, scale, causal,
                    window, reinterpret_cast<cudaStream_t>(stream), dev->err);
}

int attn_decode_splitkv_fp8(const void* q, const void* k_cache, const void* v_cache, float k_scale,
                            float v_scale, const int* seqlens, void* workspace, int B, int Hq,
                            int Hkv, int Nk_max, int D, float scale, int chunk,
                            attn_stream_t stream) {
  if (!q || !k_cache || !v_cache || !seqlens || !workspace) return ATTN_ERR_NULL;
  int rc = check_decode(B, Hq, Hkv, Nk_max, D, chunk);
  if (rc != ATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace) ||
      !aligned16(seqlens))
    return ATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f) || !std::isfinite(k_scale) || !(k_scale > 0.f) ||
      !std::isfinite(v_scale) || !(v_scale > 0.f))
    return ATTN_ERR_SCALE;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return launch_decode_splitkv(q, k_cache, v_cache, seqlens, workspace, B, Hq, Hkv, Nk_max, D, scale,
                               chunk, dev->num_sms, reinterpret_cast<cudaStream_t>(stream), dev->err,
                               1, k_scale, v_scale);
}

int attn_decode_splitkv_paged_fp8(const void* q, const void* k_pages, const void* v_pages,
                                  float k_scale, float v_scale, const int* block_table,
                                  const int* seqlens, void* workspace, int B, int Hq, int Hkv,
                                  int num_pages, int page_size, int max_pages, int D, float scale,
                                  int chunk, attn_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !seqlens || !workspace) return ATTN_ERR_NULL;
  if (num_pages <= 0 || max_pages <= 0 || page_size <= 0 || page_size % 64 != 0) return ATTN_ERR_DIM;
  if (static_cast<long long>(max_pages) * page_size > 0x7fffffffLL) return ATTN_ERR_DIM;
  int rc = check_decode(B, Hq, Hkv, max_pages * page_size, D, chunk);
  if (rc != ATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(workspace) ||
      !aligned16(seqlens) || !aligned16(block_table))
    return ATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f) || !std::isfinite(k_scale) || !(k_scale > 0.f) ||
      !std::isfinite(v_scale) || !(v_scale > 0.f))
    return ATTN_ERR_SCALE;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return launch_decode_splitkv_paged(q, k_pages, v_pages, block_table, seqlens, workspace, B, Hq,
                                     Hkv, num_pages, page_size, max_pages, D, scale, chunk,
                                     dev->num_sms, reinterpret_cast<cudaStream_t>(stream), dev->err,
                                     1, k_scale, v_scale);
}

int attn_decode_combine(const void* workspace, const int* seqlens, void* o, float* lse, int B,
                        int Hq, int Nk_max, int D, int chunk, attn_stream_t stream) {
  if (!workspace || !seqlens || !o) return ATTN_ERR_NULL;
  int rc = check_decode(B, Hq, Hq, Nk_max, D, chunk);  // no KV heads involved here
  if (rc != ATTN_OK) return rc;
  if (!aligned16(workspace) || !aligned16(seqlens) || !aligned16(o) || (lse && !aligned16(lse)))
    return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != ATTN_OK) return rc;
  return (launch_decode_combine(workspace, seqlens, o, lse, B, Hq, Nk_max, D, chunk,
                                      reinterpret_cast<cudaStream_t>(stream), dev->err));
}

int attn_get_device_error(attn_stream_t stream) {
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != ATTN_OK) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, dev->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return word;
}

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_DIM: return "a size is non-positive or too large";
    case ATTN_ERR_GQA: return "Hq is not a supported multiple of Hkv";
    case ATTN_ERR_HEAD_DIM: return "head dimension not supported by this entry point";
    case ATTN_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case ATTN_ERR_SCALE: return "scale is not finite and positive";
    case ATTN_ERR_CUDA: return "CUDA runtime or launch error";
    case ATTN_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case ATTN_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case ATTN_ERR_SEQLEN: return "a decode sequence length is outside [1, Nk_max]";
    case ATTN_ERR_CHUNK: return "split-KV chunk must be a multiple of 64 in [64, 1024]";
    case ATTN_ERR_CAPACITY: return "a size exceeds a fixed capacity of the entry point";
    case ATTN_ERR_PAGE: return "a block-table entry in use is outside [0, num_pages)";
    default: return "unknown status code";
  }
}

}  // extern "C"

// attn_decode_noalloc.cu — split-KV decode for callers that cannot allocate
// device memory.
//
// The regular decode entry points need a caller-provided workspace for the
// per-chunk partial results.  Some callers cannot provide one: a plugin that
// runs inside a host runtime which owns the whole device memory pool and gives
// its plugins no allocator, or a latency-critical caller that must never reach
// cudaMalloc (which can synchronise the device).  attn_decode_noalloc serves
// them: it runs the same partial and combine kernels, but keeps the partials
// in a scratch array that is part of the library image itself, so the caller
// passes only its inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// part of the library holds its kScratchBytes until the process exits.  In
// host code the array's name is only a host-side stand-in, so the device
// address is fetched with cudaGetSymbolAddress once per device (with that
// device current) on the first call there, and passed to the kernels.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"

namespace {

constexpr size_t kScratchBytes = ATTN_DECODE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (major != 10 || minor != 3) return ATTN_ERR_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return ATTN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                   const int* seqlens, void* o, float* lse, int B, int Hq,
                                   int Hkv, int Nk_max, int D, float scale, int chunk,
                                   attn_stream_t stream) {
  if (!q || !k_cache || !v_cache || !seqlens || !o) return ATTN_ERR_NULL;
  const size_t need = attn_decode_workspace_size(B, Hq, D, Nk_max, chunk);
  if (need == 0) return ATTN_ERR_DIM;
  if (need > kScratchBytes) return ATTN_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(o) & 15u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 15u)))
    return ATTN_ERR_ALIGN;
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != ATTN_OK) return rc;
  // The partial step writes every (b, h, chunk) entry that the combine step
  // reads, so nothing left in the scratch by an earlier call is ever used.
  rc = attn_decode_splitkv(q, k_cache, v_cache, seqlens, scratch, B, Hq, Hkv, Nk_max, D, scale,
                           chunk, stream);
  if (rc != ATTN_OK) return rc;
  return attn_decode_combine(scratch, seqlens, o, lse, B, Hq, Nk_max, D, chunk, stream);
}

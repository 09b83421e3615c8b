// Test-only kernel: exercises the library's bounded mbarrier wait (ptx.cuh)
// on a barrier that nothing ever arrives on.  Warp 0 must give up after the
// wait limit, set ATTN_ERR_TIMEOUT in the error word and raise the CTA's abort
// flag; warp 1, waiting on the same barrier, must then stop through the abort
// flag.  No fault, trap or unbounded loop is involved.
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace {

__global__ void wait_timeout_probe_kernel(int* err, int* result, unsigned long long* elapsed_ns) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  const uint32_t b = attn::smem_u32(&bar);
  if (threadIdx.x == 0) {
    attn::mbar_init(b, 1);
    abort_flag = 0;
    attn::fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x / 32;
  if ((threadIdx.x & 31) == 0) {
    const unsigned long long t0 = attn::global_ns();
    const bool ok = attn::mbar_wait(b, 0, reinterpret_cast<volatile int*>(&abort_flag), err);
    result[warp] = ok ? 1 : 0;
    elapsed_ns[warp] = attn::global_ns() - t0;
  }
}

}  // namespace

extern "C" int wait_timeout_probe(int* err, int* result, unsigned long long* elapsed_ns) {
  wait_timeout_probe_kernel<<<1, 64>>>(err, result, elapsed_ns);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -2;
}

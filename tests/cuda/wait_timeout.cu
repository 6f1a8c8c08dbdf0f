// Test-only kernel for the bounded-wait failure path of the library's
// mbarrier wait (blackwell_programming_gb300/csrc/ptx.cuh).  Nothing ever
// arrives on the barriers, so warp 0's wait gives up after the library's
// limit, records where in the error word and raises the CTA's abort flag;
// warp 1 starts waiting later and must return through the abort flag long
// before its own limit.  No trap and no fault: both waits just return.
#include <cstdio>

#include "../../blackwell_programming_gb300/csrc/ptx.cuh"

using namespace gbattn;

__global__ void wait_timeout_kernel(unsigned* err, unsigned long long* exit_ns, unsigned* results) {
  __shared__ __align__(8) unsigned long long bars[2];
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx w{&abort_flag, err};
  const unsigned long long t0 = globaltimer_ns();
  const uint32_t warp = threadIdx.x >> 5;
  bool ok = true;
  if (warp == 0) {
    ok = mbar_wait(smem_u32(&bars[0]), 0, w);
  } else {
    while (globaltimer_ns() - t0 < 200000000ull) {   // start 0.2 s later
    }
    ok = mbar_wait(smem_u32(&bars[1]), 0, w);
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    exit_ns[warp] = globaltimer_ns() - t0;
    results[warp] = ok ? 1u : 0u;
  }
  if (threadIdx.x == 0) results[2] = smem_u32(&bars[0]);
}

extern "C" int run_wait_timeout(unsigned* h_err, unsigned long long* h_exit_ns, unsigned* h_results) {
  unsigned* err = nullptr;
  unsigned long long* ex = nullptr;
  unsigned* res = nullptr;
  if (cudaMalloc(&err, 8 * sizeof(unsigned)) != cudaSuccess) return 1;
  if (cudaMalloc(&ex, 2 * sizeof(unsigned long long)) != cudaSuccess) return 1;
  if (cudaMalloc(&res, 4 * sizeof(unsigned)) != cudaSuccess) return 1;
  cudaMemset(err, 0, 8 * sizeof(unsigned));
  wait_timeout_kernel<<<1, 64>>>(err, ex, res);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return 2;
  cudaMemcpy(h_err, err, 8 * sizeof(unsigned), cudaMemcpyDeviceToHost);
  cudaMemcpy(h_exit_ns, ex, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  cudaMemcpy(h_results, res, 4 * sizeof(unsigned), cudaMemcpyDeviceToHost);
  cudaFree(err);
  cudaFree(ex);
  cudaFree(res);
  return 0;
}

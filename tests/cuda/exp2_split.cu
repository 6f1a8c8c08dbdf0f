// Test-only kernel for the library's exponential on the FMA pipe
// (ex2_fma2 in blackwell_programming_gb300/csrc/ptx.cuh): evaluates it and
// the SFU's ex2.approx on the same arguments, so a test can bound the
// polynomial's error against the hardware exponential.
#include <cuda_runtime.h>

#include "../../blackwell_programming_gb300/csrc/ptx.cuh"

using namespace gbattn;

__global__ void exp2_both(const float* x, float* poly, float* sfu, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i + 1 >= n + 1) return;
  const float x0 = x[i], x1 = (i + 1 < n) ? x[i + 1] : 0.f;
  const uint64_t p = ex2_fma2(f2_pack(x0, x1));
  poly[i] = f2_lo(p);
  sfu[i] = ex2(x0);
  if (i + 1 < n) {
    poly[i + 1] = f2_hi(p);
    sfu[i + 1] = ex2(x1);
  }
}

// x, poly and sfu are host arrays of n floats; returns a cudaError_t.
extern "C" int run_exp2_both(const float* x, float* poly, float* sfu, int n) {
  float *dx = nullptr, *dp = nullptr, *ds = nullptr;
  const size_t bytes = static_cast<size_t>(n) * sizeof(float);
  cudaError_t e;
  if ((e = cudaMalloc(&dx, bytes)) != cudaSuccess) return e;
  if ((e = cudaMalloc(&dp, bytes)) != cudaSuccess) return e;
  if ((e = cudaMalloc(&ds, bytes)) != cudaSuccess) return e;
  cudaMemcpy(dx, x, bytes, cudaMemcpyHostToDevice);
  const int pairs = (n + 1) / 2;
  exp2_both<<<(pairs + 255) / 256, 256>>>(dx, dp, ds, n);
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return e;
  cudaMemcpy(poly, dp, bytes, cudaMemcpyDeviceToHost);
  cudaMemcpy(sfu, ds, bytes, cudaMemcpyDeviceToHost);
  cudaFree(dx);
  cudaFree(dp);
  cudaFree(ds);
  return cudaGetLastError();
}

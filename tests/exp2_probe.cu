// Test probe: evaluates the prefill softmax's FMA-pipe 2^x (pkv_exp2.cuh) next to
// CUDA's exp2f on the same inputs.  Built and called by tests/test_exp2_fma.py only.
#include <cuda_runtime.h>

#include "pkv_exp2.cuh"

__global__ void exp2_probe_kernel(const float *x, float *poly, float *ref, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    poly[i] = pkv::dev::exp2_fma(x[i]);
    ref[i] = exp2f(x[i]);
  }
}

extern "C" int exp2_probe(const float *x, float *poly, float *ref, int n) {
  if (n <= 0) return 0;
  exp2_probe_kernel<<<(n + 255) / 256, 256>>>(x, poly, ref, n);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}

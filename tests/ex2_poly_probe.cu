// Test-only kernel (built by tests/test_exp2_device.py, not part of the
// library): evaluates the softmax's FMA-pipe exp2, attn::ex2_poly2, on an
// array of inputs so that the test can compare it with 2^x in float64.
#include <cuda_runtime.h>

#include "attn_device.cuh"

__global__ void ex2_poly_eval(const float* x, float* y, int n) {
  const int i = 2 * static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
  if (i + 1 < n) {
    float a = x[i], b = x[i + 1];
    attn::ex2_poly2(a, b);
    y[i] = a;
    y[i + 1] = b;
  }
}

// n must be even; x and y are device arrays of n floats.
extern "C" int ex2_poly_eval_launch(const float* x, float* y, int n, cudaStream_t stream) {
  if (n <= 0 || (n & 1)) return -1;
  const int pairs = n / 2;
  ex2_poly_eval<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y, n);
  return static_cast<int>(cudaGetLastError());
}

// Test-only kernel (built by tests/test_tmem_ldred_device.py, not part of the
// library): pins the semantics the FP8 kernel relies on for the reducing TMEM
// load, tcgen05.ld.red.32x32b.x32.max.f32 — each thread gets its TMEM row's
// 32 columns in registers and, in one more register, their maximum.  One CTA
// of 128 threads writes known rows into 32 TMEM columns, reads them back with
// the reducing load and returns both.
#include <cuda_runtime.h>

#include "attn_device.cuh"

__global__ void __launch_bounds__(128, 1) ldred_probe(const float* in, float* vals, float* maxes) {
  __shared__ uint32_t slot;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    attn::tmem_alloc(attn::smem_u32(&slot), 32);
    attn::tmem_relinquish();
    attn::tc_fence_before();
  }
  __syncthreads();
  attn::tc_fence_after();
  const uint32_t t = slot + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's 32 lanes
  const int r = threadIdx.x;                                          // TMEM lane = row
  uint32_t w[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(in[r * 32 + c]);
  attn::tmem_st32(t, w);
  attn::tmem_wait_st();
  uint32_t v[32];
  float m;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
        "=f"(m)
      : "r"(t));
  attn::tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < 32; ++c) vals[r * 32 + c] = __uint_as_float(v[c]);
  maxes[r] = m;
  attn::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    attn::tc_fence_after();
    attn::tmem_dealloc(slot, 32);
  }
}

// in: 128 × 32 floats (row r = TMEM lane r); vals the same shape; maxes 128.
extern "C" int ldred_probe_launch(const float* in, float* vals, float* maxes, cudaStream_t stream) {
  ldred_probe<<<1, 128, 0, stream>>>(in, vals, maxes);
  return static_cast<int>(cudaGetLastError());
}

// tcgen05.mma throughput microbenchmark for sm_103a (not part of the library).
//
// One CTA per SM (152).  NT threads, each in its own warp, issue ITERS MMAs
// of shape 128 × N × 16 (kind::f16, bf16 operands, fp32 accumulate) into
// their own TMEM columns, A and B from shared memory (SS) or A from TMEM (TS),
// then commit and wait; the time from first issue to completion, in SM
// clocks, gives cycles per MMA for the CTA.  Optionally eight more warps load
// the SM meanwhile: LOAD bit 0 — TMEM loads and stores (as the softmax
// warps do), bit 1 — MUFU exp2 and FMA work.  Operand tiles are zero; every
// wait is bounded.
//
// Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o /tmp/mma_rates \
//        exact_attention_63_gb300/microbench/mma_rates.cu && /tmp/mma_rates
#include <cstdio>
#include <cstdlib>

#include "../csrc/attn_device.cuh"

using namespace attn;

constexpr int kIters = 4096;
constexpr int kLoadWarps = 8;
constexpr int kThreads = (4 + kLoadWarps) * 32;

template <int N, int NT, bool TS, int LOAD>
__global__ void __launch_bounds__(kThreads, 1) mma_rates(unsigned long long* out) {
  static_assert(NT >= 1 && NT <= 4 && NT * N <= 256, "accumulators must fit in columns [0, 256)");
  extern __shared__ uint8_t dyn[];
  __shared__ uint32_t slot;
  __shared__ __align__(8) uint64_t bar[4];
  __shared__ volatile uint32_t issuers_left;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(dyn), base = (raw + 1023u) & ~1023u;
  if (warp == 0) {
    tmem_alloc(smem_u32(&slot), 512);
    tmem_relinquish();
  }
  if (threadIdx.x < 4) mbar_init(smem_u32(&bar[threadIdx.x]), 1);
  if (threadIdx.x == 0) issuers_left = NT;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  for (int i = threadIdx.x; i < 2 * 16384 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(dyn + (base - raw))[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot;
  if (warp < NT) {
    if (lane == 0) {
      const uint64_t dA = sdesc_kmajor_sw128(base), dB = sdesc_kmajor_sw128(base + 16384);
      constexpr uint32_t id = idesc_bf16(128, N, false);
      const uint32_t tacc = tmem + N * warp;  // columns [N·warp, N·warp + N)
      const uint32_t tA = tmem + 384;         // TS operand: columns [384, 392)
      const unsigned long long t0 = clock64();
      for (int i = 0; i < kIters; ++i) {
        const uint32_t off = ((i & 3) * 32) >> 4;  // K step within the 128-byte swizzle row
        if (TS)
          mma_ts(tacc, tA, dB + off, id, i > 0 ? 1u : 0u);
        else
          mma_ss(tacc, dA + off, dB + off, id, i > 0 ? 1u : 0u);
      }
      mma_commit(smem_u32(&bar[warp]));
      const uint64_t g0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&bar[warp]), 0))
        if (globaltimer_ns() - g0 > 2000000000ull) break;
      out[blockIdx.x * 4 + warp] = clock64() - t0;
      atomicSub(const_cast<uint32_t*>(&issuers_left), 1u);
    }
  } else if (warp >= 4 && LOAD != 0) {
    // Load warps: TMEM traffic in columns [256, 384) and/or exp2 + FMA work,
    // until every issuer has finished (bounded).
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tcol = tmem + 256 + 64 * ((warp - 4) >> 2);
    float acc = 0.25f * lane;
    for (int it = 0; it < (1 << 20) && issuers_left != 0; ++it) {
      uint32_t v[32];
      if (LOAD & 1) {
        tmem_ld32(tcol + lane_off, v);
        tmem_wait_ld();
        reg_fence32(v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(acc + i);
      }
      if (LOAD & 2) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(ex2_mufu(__uint_as_float(v[i]) * 0.01f - 1.f) * 0.5f + acc);
      }
      if (LOAD & 1) {
        tmem_st32(tcol + lane_off, v);
        tmem_wait_st();
      }
      acc += __uint_as_float(v[it & 31]) * 1e-30f;
    }
    if (acc == 12345.f) out[152 * 4] = 1;  // keeps the work live
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int N, int NT, bool TS, int LOAD>
void run(unsigned long long* d, const char* note) {
  constexpr int smem = 2 * 16384 + 1024;
  if (cudaFuncSetAttribute(mma_rates<N, NT, TS, LOAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess) {
    std::printf("attribute error\n");
    std::exit(1);
  }
  cudaMemset(d, 0, (152 * 4 + 1) * 8);
  mma_rates<N, NT, TS, LOAD><<<152, kThreads, smem>>>(d);
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    std::printf("error %s\n", cudaGetErrorString(e));
    std::exit(1);
  }
  unsigned long long h[152 * 4];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  double mx = 0;
  for (int b = 0; b < 152; ++b)
    for (int t = 0; t < NT; ++t) mx = h[b * 4 + t] > mx ? h[b * 4 + t] : mx;
  const double per = mx / (static_cast<double>(kIters) * NT);  // cycles per MMA for the CTA
  std::printf("| %s, N=%d, %d issuing thread%s%s | %.1f | %.0f |\n", TS ? "TS" : "SS", N, NT, NT > 1 ? "s" : "",
              note, per, 2.0 * 128 * N * 16 / per);
}

int main() {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, (152 * 4 + 1) * 8) != cudaSuccess) return 1;
  std::printf("| variant (M=128, K=16) | cycles per MMA | FLOP/clk/SM |\n|---|---|---|\n");
  run<128, 1, false, 0>(d, "");
  run<128, 2, false, 0>(d, "");
  run<64, 1, false, 0>(d, "");
  run<64, 2, false, 0>(d, "");
  run<64, 4, false, 0>(d, "");
  run<32, 4, false, 0>(d, "");
  run<128, 1, true, 0>(d, "");
  run<64, 1, true, 0>(d, "");
  run<64, 2, true, 0>(d, "");
  run<64, 4, true, 0>(d, "");
  run<128, 1, false, 1>(d, " + 8 warps of TMEM loads/stores");
  run<128, 1, false, 2>(d, " + 8 warps of exp2/FMA work");
  run<128, 1, false, 3>(d, " + 8 warps doing both");
  cudaFree(d);
  return 0;
}

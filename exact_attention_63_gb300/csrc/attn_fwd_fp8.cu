// Attention forward kernels for FP8 (E4M3) inputs, head dim 128, full and causal masks.
#include "attn_fwd_fp8.cuh"
#include "attn_launch.h"

namespace attn {

template <bool CAUSAL>
static cudaError_t launch_fp8_one(const LaunchArgs& a) {
  constexpr unsigned int smem = Fp8Layout::kSmemBytes;
  static volatile bool configured[64] = {};
  if (a.device < 0 || a.device >= 64) return cudaErrorInvalidDevice;
  if (!configured[a.device]) {
    const cudaError_t e =
        cudaFuncSetAttribute(attn_fwd_fp8_kernel<CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[a.device] = true;
  }
  attn_fwd_fp8_kernel<CAUSAL><<<a.grid, kThreads, smem, a.stream>>>(a.q, a.k, a.v, a.o, a.p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const LaunchArgs& a, bool causal) {
  return causal ? launch_fp8_one<true>(a) : launch_fp8_one<false>(a);
}

}  // namespace attn

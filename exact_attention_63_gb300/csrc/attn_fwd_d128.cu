// Instantiations of the attention forward kernel for head dim 128.
#include "attn_launch.h"

namespace attn {
namespace {

template <bool CAUSAL>
cudaError_t launch_impl(const LaunchArgs& a) {
  constexpr unsigned int smem = Layout<128>::kSmemBytes;
  // The dynamic shared-memory opt-in is per device and per kernel; set it the
  // first time each device launches this instantiation.
  static volatile bool configured[64] = {};
  if (a.device < 0 || a.device >= 64) return cudaErrorInvalidDevice;
  if (!configured[a.device]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<128, CAUSAL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[a.device] = true;
  }
  attn_fwd_kernel<128, CAUSAL><<<a.grid, kThreads, smem, a.stream>>>(a.q, a.k, a.v, a.o, a.p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d128(const LaunchArgs& a) {
  return a.causal ? launch_impl<true>(a) : launch_impl<false>(a);
}

}  // namespace attn

// Attention forward kernels for FP8 (E4M3) inputs, head dim 128, full and causal masks.
#include "attn_fwd_fp8.cuh"
#include "attn_fwd_fp8_rows.cuh"
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

// The full-row kernel (two CTAs per SM).  Its register split relies on the
// kernel being compiled to exactly kFp8RowsLaunchRegs registers; a build where
// it is not runs the one-CTA kernel instead (cudaErrorNotSupported).
template <bool CAUSAL>
static cudaError_t launch_fp8_rows_one(const LaunchArgs& a) {
  constexpr unsigned int smem = Fp8RowsLayout::kSmemBytes;
  static volatile int state[64] = {};  // per device: 0 not checked, 1 usable, -1 not usable
  if (a.device < 0 || a.device >= 64) return cudaErrorInvalidDevice;
  if (state[a.device] == 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_fwd_fp8_rows_kernel<CAUSAL>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kFp8RowsLaunchRegs) {
      state[a.device] = -1;
    } else {
      e = cudaFuncSetAttribute(attn_fwd_fp8_rows_kernel<CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      state[a.device] = 1;
    }
  }
  if (state[a.device] < 0) return cudaErrorNotSupported;
  const int grid = a.p.n_tiles < 2 * a.sms ? a.p.n_tiles : 2 * a.sms;
  attn_fwd_fp8_rows_kernel<CAUSAL><<<grid, kFp8RowsThreads, smem, a.stream>>>(a.q, a.k, a.v, a.o, a.p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const LaunchArgs& a, bool causal) {
  if (!(a.p.test_flags & ATTN_TEST_FALLBACK_KERNEL)) {
    const cudaError_t e = causal ? launch_fp8_rows_one<true>(a) : launch_fp8_rows_one<false>(a);
    if (e != cudaErrorNotSupported) return e;
  }
  return causal ? launch_fp8_one<true>(a) : launch_fp8_one<false>(a);
}

}  // namespace attn

// Attention backward kernels: instantiations and launches (both head dims,
// both masks, the two passes and the one-pass kernel at d = 64), the preparation
// kernel and the rounding of the one-pass kernel's dQ.
#include "attn_bwd_launch.h"

#include "attn_bwd_kernel.cuh"

namespace attn {
namespace {

template <int D, bool CAUSAL, int MODE>
cudaError_t launch_bwd_one(const BwdLaunchArgs& a) {
  constexpr unsigned int smem = BwdLayout<D, MODE>::kSmemBytes;
  static volatile bool configured[64] = {};
  if (a.device < 0 || a.device >= 64) return cudaErrorInvalidDevice;
  if (!configured[a.device]) {
    const cudaError_t e =
        cudaFuncSetAttribute(attn_bwd_kernel<D, CAUSAL, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[a.device] = true;
  }
  attn_bwd_kernel<D, CAUSAL, MODE><<<a.grid, kBwdThreads, smem, a.stream>>>(a.x, a.x2, a.a, a.b, a.o0, a.o1, a.dq,
                                                                             a.p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_d(const BwdLaunchArgs& a) {
  if (a.mode == kModeDQ)
    return a.causal ? launch_bwd_one<D, true, kModeDQ>(a) : launch_bwd_one<D, false, kModeDQ>(a);
  if (a.mode == kModeFused) {
    // The one-pass kernel is built for d = 64 only: at d = 128 its dQ
    // reduce-adds run into the L2's reduction rate and the two passes are
    // faster.
    if constexpr (D == 64)
      return a.causal ? launch_bwd_one<D, true, kModeFused>(a) : launch_bwd_one<D, false, kModeFused>(a);
    else
      return cudaErrorInvalidValue;
  }
  return a.causal ? launch_bwd_one<D, true, kModeDKV>(a) : launch_bwd_one<D, false, kModeDKV>(a);
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunchArgs& a, int d) {
  if (d == 64) return launch_bwd_d<64>(a);
  if (d == 128) return launch_bwd_d<128>(a);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_prep(const void* o, const long long o_st[3], const void* dout, const float* lse, float* lse2,
                            float* dvec, float* dq_acc, int B, int H, int Sq, int pitch, int d, cudaStream_t stream) {
  const long long n = static_cast<long long>(B) * H * pitch;  // rows, 32·8/d per warp
  const int threads = 256;
  const long long want = n * d / (8 * 32 * (threads / 32)) + 1;
  const int blocks = static_cast<int>(want < 16384 ? want : 16384);
  const uint16_t* o16 = static_cast<const uint16_t*>(o);
  const uint16_t* g16 = static_cast<const uint16_t*>(dout);
  if (d == 64)
    attn_bwd_prep_kernel<64><<<blocks, threads, 0, stream>>>(o16, o_st[0], o_st[1], o_st[2], g16, lse, lse2, dvec,
                                                              dq_acc, B, H, Sq, pitch);
  else
    attn_bwd_prep_kernel<128><<<blocks, threads, 0, stream>>>(o16, o_st[0], o_st[1], o_st[2], g16, lse, lse2, dvec,
                                                               dq_acc, B, H, Sq, pitch);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(const float* dq_acc, void* dq, int B, int H, int Sq, int pitch, int d, float scale,
                                  int sms, cudaStream_t stream) {
  const long long n = static_cast<long long>(B) * Sq * H * (d / 8);
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 152) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  if (d != 64) return cudaErrorInvalidValue;  // the one-pass kernel's head dim
  attn_bwd_dq_convert_kernel<64><<<blocks, threads, 0, stream>>>(dq_acc, static_cast<uint16_t*>(dq), B, H, Sq, pitch,
                                                                  scale);
  return cudaGetLastError();
}

}  // namespace attn

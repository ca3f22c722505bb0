// attn_fwd_host_static: the host-buffer attention call for callers that
// cannot allocate device memory.  The device staging area for q, k, v, o and
// lse is a fixed-size array in this library's device image.  It is reserved
// when the CUDA runtime loads this file's module on a device: with lazy
// module loading (the default) that is the first call on the device, with
// eager loading it is library load.
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "attn_gb300.h"
#include "attn_launch.h"

namespace {

constexpr size_t kStaticBytes = ATTN_STATIC_WORKSPACE_BYTES;

// Staging area of attn_fwd_host_static.  In host code this name is only a
// handle for the runtime; the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_static_workspace[kStaticBytes];

}  // namespace

extern "C" int attn_fwd_host_static(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                                    int B, int H, int Sq, int Sk, int d, float scale, int causal,
                                    cudaStream_t stream) {
  if (q_h == nullptr || k_h == nullptr || v_h == nullptr || o_h == nullptr || lse_h == nullptr) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEAD_DIM;
  const size_t need = attn_fwd_host_workspace_size(B, H, Sq, Sk, d);
  if (need == 0 || need > kStaticBytes) return ATTN_ERR_STATIC_LIMIT;

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn::record_cuda_error(e, "cudaGetDevice");
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
      minor != 3)
    return ATTN_ERR_ARCH;

  // The array's device address on the current device, looked up on every
  // call (no cache: a context torn down and re-created may place the module
  // elsewhere).  Once the module is loaded this is a host-side table lookup
  // that allocates nothing; the first lookup on a device loads the module,
  // which reserves the array and can fail with out-of-memory.
  void* addr = nullptr;
  e = cudaGetSymbolAddress(&addr, g_static_workspace);
  if (e != cudaSuccess) return attn::record_cuda_error(e, "cudaGetSymbolAddress(static workspace)");
  if (addr == nullptr) return attn::record_cuda_error(cudaErrorInvalidSymbol, "cudaGetSymbolAddress(static workspace)");
  // Every byte the kernel and the copies read back is written earlier in the
  // same call (q/k/v by the host-to-device copies, o/lse by the kernel), so
  // nothing in the array needs clearing between calls.
  // The single-slice form: it creates no streams or events either.
  return attn::fwd_host(q_h, k_h, v_h, o_h, lse_h, B, H, Sq, Sk, d, scale, causal, addr, kStaticBytes, stream,
                        false);
}

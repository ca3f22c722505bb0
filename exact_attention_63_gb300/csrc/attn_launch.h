// Internal interface between the C-ABI host code (attn_api.cu) and the
// per-head-dim kernel translation units (attn_fwd_d64.cu, attn_fwd_d128.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"

namespace attn {

struct LaunchArgs {
  CUtensorMap q, k, v, o;  // 4-D tiled maps, box (64, 1, 128, 1), 128-byte swizzle
  FwdParams p;
  int grid;
  int causal;
  int device;
  cudaStream_t stream;
};

cudaError_t launch_fwd_d64(const LaunchArgs& a);
cudaError_t launch_fwd_d128(const LaunchArgs& a);

// Dynamic shared memory each instantiation requests.
unsigned int fwd_smem_bytes(int d);

}  // namespace attn

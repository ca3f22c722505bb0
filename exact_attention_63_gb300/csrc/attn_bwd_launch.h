// Internal interface between the C-ABI host code (attn_api.cu) and the
// backward kernels' translation unit (attn_bwd.cu).
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

struct BwdParams {
  const float* lse2;   // [B·H, pitch]: −LSE · log2(e) of each query row; −inf beyond Sq
  const float* dvec;   // [B·H, pitch]: D = rowsum(dO ∘ O); 0 beyond Sq
  unsigned int* status;
  int B, H, Sq, Sk, pitch;
  int coff;            // causal: key j visible to query i iff j ≤ i + coff (may be negative)
  int group;           // query heads per key/value head (H / H_kv)
  int n_rt;            // row tiles per (batch, row head): row heads are H (dQ pass) or H_kv (dK/dV pass)
  float scale_log2;    // scale · log2(e)
  float scale;
  uint64_t timeout_ns;
};

struct BwdLaunchArgs {
  CUtensorMap x, x2, a, b;  // row tiles X, X2 and the streamed A, B (4-D maps as in the forward)
  CUtensorMap o0, o1;       // outputs (bf16, dense): dQ pass o0 = dQ [B, Sq, H, D]; dK/dV and fused passes
                            // o0 = dV, o1 = dK [B, Sk, H_kv, D]
  CUtensorMap dq;           // fused pass: fp32 dQ accumulator [B·H·pitch, D], box 32 × 32, 128-byte swizzle
  BwdParams p;
  int grid;
  int mode;                 // 0: dQ pass, 1: dK/dV pass, 2: fused (dK, dV and the dQ accumulator)
  bool causal;
  int device;
  cudaStream_t stream;
};

cudaError_t launch_bwd(const BwdLaunchArgs& a, int d);
// o_st: o's element strides (batch, sequence, head; d contiguous; dout is
// dense).  dq_acc: the fused pass's accumulator [B·H, pitch, d] (zeroed here),
// or null.
cudaError_t launch_bwd_prep(const void* o, const long long o_st[3], const void* dout, const float* lse, float* lse2,
                            float* dvec, float* dq_acc, int B, int H, int Sq, int pitch, int d, cudaStream_t stream);
// dq [B, Sq, H, d] bf16 = scale · dq_acc [B·H, pitch, d].
cudaError_t launch_bwd_dq_convert(const float* dq_acc, void* dq, int B, int H, int Sq, int pitch, int d, float scale,
                                  int sms, cudaStream_t stream);

}  // namespace attn

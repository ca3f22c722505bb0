// Internal interface between the C-ABI host code (attn_api.cu) and the
// kernel translation units (one per head dim × mask kind).
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"
#include "attn_fwd_rows.cuh"
#include "attn_gb300.h"

namespace attn {

struct LaunchArgs {
  CUtensorMap q, k, v, o;  // 4-D tiled maps, box (64, 1, 128, 1), 128-byte swizzle
  FwdParams p;
  int grid;             // persistent: min(tiles, SMs)
  int sms;              // multiprocessors of the device
  uint32_t poly;           // exp2 chunk mask; one of kPolyMasks
  int device;
  cudaStream_t stream;
};

// The exp2 splits compiled into the library (bit c = 16-column chunk c of a
// 128-key block uses the polynomial): none, 1/8, 1/4, 1/2, all.
constexpr uint32_t kPolyMasks[] = {0x00u, 0x01u, 0x11u, 0x55u, 0xFFu};

inline bool poly_mask_supported(uint32_t m) {
  for (uint32_t x : kPolyMasks)
    if (x == m) return true;
  return false;
}

// attn_fwd_host with or without the chunked copy/compute pipeline (the
// single-slice form uses only the caller's stream and creates no streams or
// events: attn_fwd_host_static uses it).
int fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h, int B, int H, int Sq, int Sk,
             int d, float scale, int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream,
             bool pipelined);

// Record a failed CUDA call for attn_last_cuda_error(); returns ATTN_ERR_LAUNCH.
int record_cuda_error(cudaError_t e, const char* what);

// FP8 (E4M3) inputs, d = 128 (attn_fwd_fp8.cu).
cudaError_t launch_fwd_fp8(const LaunchArgs& a, bool causal);

cudaError_t launch_fwd_d64(const LaunchArgs& a);
cudaError_t launch_fwd_d64_causal(const LaunchArgs& a);
cudaError_t launch_fwd_d128(const LaunchArgs& a);
cudaError_t launch_fwd_d128_causal(const LaunchArgs& a);

// Launch one instantiation, setting its shared-memory opt-in the first time
// each device uses it.
template <int D, bool CAUSAL, uint32_t POLY, bool COUNT, bool VARLEN>
cudaError_t launch_one(const LaunchArgs& a) {
  constexpr unsigned int smem = Layout<D>::kSmemBytes + (VARLEN && !CAUSAL ? kSeqTableBytes : 0u);
  static volatile bool configured[64] = {};
  if (a.device < 0 || a.device >= 64) return cudaErrorInvalidDevice;
  if (!configured[a.device]) {
    const cudaError_t e =
        cudaFuncSetAttribute(attn_fwd_kernel<D, CAUSAL, POLY, COUNT, VARLEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    configured[a.device] = true;
  }
  attn_fwd_kernel<D, CAUSAL, POLY, COUNT, VARLEN><<<a.grid, kThreads, smem, a.stream>>>(a.q, a.k, a.v, a.o, a.p);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool COUNT>
cudaError_t launch_poly(const LaunchArgs& a) {
  switch (a.poly) {
    case 0x00u: return launch_one<D, CAUSAL, 0x00u, COUNT, false>(a);
    case 0x01u: return launch_one<D, CAUSAL, 0x01u, COUNT, false>(a);
    case 0x11u: return launch_one<D, CAUSAL, 0x11u, COUNT, false>(a);
    case 0x55u: return launch_one<D, CAUSAL, 0x55u, COUNT, false>(a);
    case 0xFFu: return launch_one<D, CAUSAL, 0xFFu, COUNT, false>(a);
    default: return cudaErrorInvalidValue;
  }
}

// The d = 64 full-row kernel (two CTAs per SM).  Its register split relies on
// the kernel being compiled to exactly kRowsLaunchRegs registers; a build
// where it is not runs the two-warpgroup kernel instead (cudaErrorNotSupported
// tells the caller to).
template <bool CAUSAL, bool COUNT, uint32_t POLY, bool VARLEN = false>
cudaError_t launch_rows_one(const LaunchArgs& a) {
  constexpr unsigned int smem = (VARLEN && !CAUSAL) ? RowsLayout::kSmemBytesTable : RowsLayout::kSmemBytes;
  static volatile int state[64] = {};  // per device: 0 not checked, 1 usable, -1 not usable
  if (a.device < 0 || a.device >= 64) return cudaErrorInvalidDevice;
  if (state[a.device] == 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_fwd_rows_kernel<CAUSAL, COUNT, POLY, VARLEN>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRowsLaunchRegs) {
      state[a.device] = -1;
    } else {
      e = cudaFuncSetAttribute(attn_fwd_rows_kernel<CAUSAL, COUNT, POLY, VARLEN>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      state[a.device] = 1;
    }
  }
  if (state[a.device] < 0) return cudaErrorNotSupported;
  const int grid = a.p.n_tiles < 2 * a.sms ? a.p.n_tiles : 2 * a.sms;
  attn_fwd_rows_kernel<CAUSAL, COUNT, POLY, VARLEN><<<grid, kRowsThreads, smem, a.stream>>>(a.q, a.k, a.v, a.o, a.p);
  return cudaGetLastError();
}

template <bool CAUSAL, bool COUNT>
cudaError_t launch_rows(const LaunchArgs& a) {
  switch (a.poly) {
    case 0x00u: return launch_rows_one<CAUSAL, COUNT, 0x00u>(a);
    case 0x01u: return launch_rows_one<CAUSAL, COUNT, 0x01u>(a);
    case 0x11u: return launch_rows_one<CAUSAL, COUNT, 0x11u>(a);
    case 0x55u: return launch_rows_one<CAUSAL, COUNT, 0x55u>(a);
    case 0xFFu: return launch_rows_one<CAUSAL, COUNT, 0xFFu>(a);
    default: return cudaErrorInvalidValue;
  }
}

// The counting kernels are separate instantiations, so the default ones carry
// no diagnostic code.  Packed sequences (offset tables given) have their own
// instantiations, compiled with the default exp2 split only.
template <int D, bool CAUSAL>
cudaError_t launch_variant(const LaunchArgs& a) {
  if (a.p.cu_q != nullptr) {
    if (a.poly != 0x00u) return cudaErrorInvalidValue;
    if (D == 64 && !(a.p.test_flags & ATTN_TEST_FALLBACK_KERNEL)) {  // the full-row kernel
      const cudaError_t e = a.p.counters != nullptr ? launch_rows_one<CAUSAL, true, 0x00u, true>(a)
                                                    : launch_rows_one<CAUSAL, false, 0x00u, true>(a);
      if (e != cudaErrorNotSupported) return e;
    }
    return a.p.counters != nullptr ? launch_one<D, CAUSAL, 0x00u, true, true>(a)
                                   : launch_one<D, CAUSAL, 0x00u, false, true>(a);
  }
  if (D == 64 && !(a.p.test_flags & ATTN_TEST_FALLBACK_KERNEL)) {  // dense tensors: the full-row kernel
    const cudaError_t e = a.p.counters != nullptr ? launch_rows<CAUSAL, true>(a) : launch_rows<CAUSAL, false>(a);
    if (e != cudaErrorNotSupported) return e;
  }
  return a.p.counters != nullptr ? launch_poly<D, CAUSAL, true>(a) : launch_poly<D, CAUSAL, false>(a);
}

}  // namespace attn

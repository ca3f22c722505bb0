// C ABI of the attention forward library: argument checks, TMA descriptor
// encoding, kernel dispatch and the device status word.  Declarations and
// their contracts are in include/attn_gb300.h.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "attn_bwd_launch.h"
#include "attn_gb300.h"
#include "attn_launch.h"

namespace {

constexpr int kMaxDevices = 64;

// One status word per device (module-scope device variable: every device that
// loads the library gets its own copy).  Kernels OR error bits into it.
__device__ unsigned int g_attn_status;

thread_local char t_last_error[256] = "";

int fail_cuda(cudaError_t e, const char* what) {
  std::snprintf(t_last_error, sizeof(t_last_error), "%s: %s", what, cudaGetErrorString(e));
  return ATTN_ERR_LAUNCH;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 4-D map over a bf16 [B, S, H, d] tensor with element strides st = (batch,
// seq, head) and contiguous d, dims innermost first (d, H, S, B); box
// (64, 1, 128, 1) = one 128-row × 128-byte slab.
int encode_bshd(CUtensorMap* m, const void* ptr, int B, int S, int H, int d, const long long st[3]) {
  auto enc = get_encode_fn();
  if (enc == nullptr) {
    std::snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled unavailable");
    return ATTN_ERR_LAUNCH;
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                                 static_cast<cuuint64_t>(st[0]) * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled failed (CUresult %d)",
                  static_cast<int>(r));
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

// 4-D map over an 8-bit [B, S, H, d] tensor, dense, dims innermost first
// (d, H, S, B); box (d, 1, 128, 1): one 128-row slab of d-byte rows (d = 128:
// exactly one 128-byte swizzle row).
int encode_bshd_u8(CUtensorMap* m, const void* ptr, int B, int S, int H, int d) {
  auto enc = get_encode_fn();
  if (enc == nullptr) {
    std::snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled unavailable");
    return ATTN_ERR_LAUNCH;
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H) * d,
                                 static_cast<cuuint64_t>(S) * H * d};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(d), 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled failed (CUresult %d)",
                  static_cast<int>(r));
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

struct DeviceInfo {
  int checked = 0;  // 0 unknown, 1 supported, -1 unsupported
  unsigned int* status = nullptr;
  int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];

int current_device(int* dev_out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    if (e != cudaSuccess) fail_cuda(e, "cudaGetDevice");
    return ATTN_ERR_ARCH;
  }
  DeviceInfo& di = g_dev[dev];
  if (di.checked == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_ARCH;
    if (major != 10 || minor != 3) {
      di.checked = -1;
    } else {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_attn_status);
      if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(status)");
      di.status = static_cast<unsigned int*>(addr);
      if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || di.sms < 1)
        return ATTN_ERR_ARCH;
      di.checked = 1;
    }
  }
  if (di.checked < 0) return ATTN_ERR_ARCH;
  *dev_out = dev;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rows that see no key (bottom-right causal alignment with Sq > Sk): O = 0,
// LSE = −inf.  One thread per (batch, head, row); rows are 16-byte aligned
// (strides are multiples of 8 elements).
__global__ void fill_unseen_rows(uint16_t* o, long long sb, long long ss, long long sh, float* lse, int lse_pitch,
                                 int B, int H, int rows, int d) {
  const long long n = static_cast<long long>(B) * H * rows;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(t % rows);
    const int h = static_cast<int>((t / rows) % H);
    const int b = static_cast<int>(t / (static_cast<long long>(rows) * H));
    uint4* row = reinterpret_cast<uint4*>(o + b * sb + i * ss + h * sh);
    for (int c = 0; c < d / 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
    lse[(static_cast<long long>(b) * H + h) * lse_pitch + i] = -INFINITY;
  }
}

// A layout's strides: all zero → dense; else each a positive multiple of 8
// elements below 2^38 (TMA: 16-byte multiples, strides below 2^40 bytes).
bool resolve_strides(const long long in[3], long long dense0, long long dense1, long long dense2, long long out[3]) {
  if (in[0] == 0 && in[1] == 0 && in[2] == 0) {
    out[0] = dense0;
    out[1] = dense1;
    out[2] = dense2;
    return true;
  }
  for (int i = 0; i < 3; ++i) {
    if (in[i] <= 0 || (in[i] & 7) != 0 || in[i] >= (1LL << 38)) return false;
    out[i] = in[i];
  }
  return true;
}

int check_args(const void* q, const void* k, const void* v, const void* o, const void* lse, int B, int H, int Sq,
               int Sk, int d, float scale) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_SHAPE;
  const long long n_qt = (static_cast<long long>(Sq) + 127) / 128;
  if (static_cast<long long>(B) * H * n_qt > 0x7FFFFFFFLL) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEAD_DIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

// Rescale threshold (log2 domain).  A stale reference bounds p by 2^τ; with
// τ = 32, fp32 row sums over up to 2^31 keys stay below 2^63 — far from
// overflow — while only a jump of 2^32 forces a rescale of O (measured: on
// peaky logits, τ = 8 rescales twice as often and runs 30% slower).
constexpr float kDefaultTau = 32.0f;
constexpr float kMaxTau = 64.0f;
constexpr unsigned int kDefaultTimeoutMs = 4000;

// Default polynomial-exp2 chunk masks (bit c = 16-column chunk c of a block),
// chosen by measurement on GB300 (whose MUFU unit is not the limiting pipe).
constexpr uint32_t kDefaultPolyMaskD64 = 0x00u;
constexpr uint32_t kDefaultPolyMaskD128 = 0x00u;

struct Opts {
  float tau = kDefaultTau;
  uint32_t poly = 0;
  unsigned long long* counters = nullptr;
  unsigned int timeout_ms = kDefaultTimeoutMs;
  unsigned int test_flags = 0;
};

int parse_options(const attn_options* opts, int d, Opts* out) {
  Opts r;
  r.poly = (d == 64) ? kDefaultPolyMaskD64 : kDefaultPolyMaskD128;
  if (opts != nullptr) {
    if (opts->struct_size < sizeof(attn_options)) return ATTN_ERR_OPTION;
    if (!std::isfinite(opts->rescale_threshold) || opts->rescale_threshold > kMaxTau) return ATTN_ERR_OPTION;
    if (opts->rescale_threshold < 0.f) r.tau = 0.f;
    else if (opts->rescale_threshold > 0.f) r.tau = opts->rescale_threshold;
    if (opts->poly_exp2_mask == 0x100u) r.poly = 0u;
    else if (opts->poly_exp2_mask != 0u) r.poly = opts->poly_exp2_mask;
    if (!attn::poly_mask_supported(r.poly)) return ATTN_ERR_OPTION;
    if (opts->counters != nullptr && (reinterpret_cast<uintptr_t>(opts->counters) & 7u) != 0) return ATTN_ERR_ALIGN;
    r.counters = opts->counters;
    if (opts->timeout_ms != 0) r.timeout_ms = opts->timeout_ms;
    if ((opts->test_flags & ~(ATTN_TEST_WITHHOLD_KV | ATTN_TEST_FALLBACK_KERNEL)) != 0) return ATTN_ERR_OPTION;
    r.test_flags = opts->test_flags;
  }
  *out = r;
  return ATTN_OK;
}

// Fill in the launch-wide fields and launch the kernel for (d, causal).
int launch(attn::LaunchArgs& a, const Opts& op, int dev, int d, int causal, float scale, cudaStream_t stream) {
  a.p.status = g_dev[dev].status;
  a.p.counters = op.counters;
  a.p.scale_log2 = scale * 1.4426950408889634f;
  a.p.tau = op.tau;
  a.p.sum_limit = std::exp2(op.tau);
  a.p.timeout_ns = static_cast<uint64_t>(op.timeout_ms) * 1000000ull;
  a.p.test_flags = op.test_flags;
  a.grid = a.p.n_tiles < g_dev[dev].sms ? a.p.n_tiles : g_dev[dev].sms;
  a.sms = g_dev[dev].sms;
  a.poly = op.poly;
  a.device = dev;
  a.stream = stream;
  cudaError_t e;
  if (d == 64) e = causal ? attn::launch_fwd_d64_causal(a) : attn::launch_fwd_d64(a);
  else e = causal ? attn::launch_fwd_d128_causal(a) : attn::launch_fwd_d128(a);
  if (e != cudaSuccess) return fail_cuda(e, "attention kernel launch");
  return ATTN_OK;
}

}  // namespace

namespace attn {

int record_cuda_error(cudaError_t e, const char* what) { return fail_cuda(e, what); }

namespace {

// attn_fwd_host's pipeline: up to kHostChunks slices of the problem, each
// copied in on `in`, computed on the caller's stream and copied out on `out`,
// so the copies of one slice overlap the kernel and the copies of the others
// (host→device and device→host use separate copy engines).  Created on a
// device's first call, kept for the process.
constexpr int kHostChunks = 4;
struct HostPipe {
  std::mutex mu;  // one enqueue sequence at a time (the events are reused)
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr, in_done[kHostChunks] = {}, k_done[kHostChunks] = {};
};
HostPipe g_pipe[kMaxDevices];

int make_pipe(HostPipe& hp) {
  if (hp.ready) return ATTN_OK;
  cudaError_t e;
  if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess) return fail_cuda(e, "stream");
  if ((e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess) return fail_cuda(e, "stream");
  cudaEvent_t* evs[2 + 2 * kHostChunks] = {&hp.start, &hp.end};
  for (int c = 0; c < kHostChunks; ++c) {
    evs[2 + c] = &hp.in_done[c];
    evs[2 + kHostChunks + c] = &hp.k_done[c];
  }
  for (cudaEvent_t* ev : evs)
    if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return fail_cuda(e, "event");
  hp.ready = true;
  return ATTN_OK;
}

}  // namespace

int fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h, int B, int H, int Sq, int Sk,
             int d, float scale, int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream,
             bool pipelined) {
  if (q_h == nullptr || k_h == nullptr || v_h == nullptr || o_h == nullptr || lse_h == nullptr) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEAD_DIM;
  const size_t need = attn_fwd_host_workspace_size(B, H, Sq, Sk, d);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return ATTN_ERR_WORKSPACE;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t qb = static_cast<size_t>(B) * Sq * H * d * 2, kb = static_cast<size_t>(B) * Sk * H * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * Sq * 4;
  char* w = static_cast<char*>(workspace);
  char* q_d = w;
  char* k_d = w + up(qb);
  char* v_d = w + up(qb) + up(kb);
  char* o_d = w + up(qb) + 2 * up(kb);
  char* l_d = w + 2 * up(qb) + 2 * up(kb);
  // Every argument error is reported before anything is enqueued.
  int rc = check_args(q_d, k_d, v_d, o_d, l_d, B, H, Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  const char* qh = static_cast<const char*>(q_h);
  const char* kh = static_cast<const char*>(k_h);
  const char* vh = static_cast<const char*>(v_h);
  char* oh = static_cast<char*>(o_h);
  char* lh = reinterpret_cast<char*>(lse_h);
  cudaError_t e;
  // Head slices need their LSE rows 16-byte aligned (Sq a multiple of 4).
  if (!pipelined || (B == 1 && (H == 1 || Sq % 4 != 0))) {
    // One slice, all on the caller's stream.
    if ((e = cudaMemcpyAsync(q_d, qh, qb, cudaMemcpyHostToDevice, stream)) != cudaSuccess) return fail_cuda(e, "copy q");
    if ((e = cudaMemcpyAsync(k_d, kh, kb, cudaMemcpyHostToDevice, stream)) != cudaSuccess) return fail_cuda(e, "copy k");
    if ((e = cudaMemcpyAsync(v_d, vh, kb, cudaMemcpyHostToDevice, stream)) != cudaSuccess) return fail_cuda(e, "copy v");
    rc = attn_fwd(q_d, k_d, v_d, o_d, reinterpret_cast<float*>(l_d), B, H, Sq, Sk, d, scale, causal, stream);
    if (rc != ATTN_OK) return rc;
    if ((e = cudaMemcpyAsync(oh, o_d, qb, cudaMemcpyDeviceToHost, stream)) != cudaSuccess) return fail_cuda(e, "copy o");
    if ((e = cudaMemcpyAsync(lh, l_d, lb, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
      return fail_cuda(e, "copy lse");
    return ATTN_OK;
  }
  int dev = -1;
  if ((rc = current_device(&dev)) != ATTN_OK) return rc;
  HostPipe& hp = g_pipe[dev];
  std::lock_guard<std::mutex> lock(hp.mu);
  if ((rc = make_pipe(hp)) != ATTN_OK) return rc;
  // Slices of the batch, or of the heads when B = 1 (strided 2-D copies; the
  // kernel reads the dense layout through element strides).
  const bool by_batch = B >= 2;
  const int units = by_batch ? B : H;
  const int nc = units < kHostChunks ? units : kHostChunks;
  const size_t row_b = static_cast<size_t>(H) * d * 2;  // bytes of one (b, s) row of q, k, v, o
  if ((e = cudaEventRecord(hp.start, stream)) != cudaSuccess) return fail_cuda(e, "record");
  if ((e = cudaStreamWaitEvent(hp.in, hp.start, 0)) != cudaSuccess) return fail_cuda(e, "wait");
  if ((e = cudaStreamWaitEvent(hp.out, hp.start, 0)) != cudaSuccess) return fail_cuda(e, "wait");
  rc = ATTN_OK;
  for (int c = 0; c < nc && rc == ATTN_OK; ++c) {
    const int u0 = static_cast<int>(static_cast<long long>(units) * c / nc);
    const int nu = static_cast<int>(static_cast<long long>(units) * (c + 1) / nc) - u0;
    size_t qo, ko, lo, ls;  // byte offsets of the slice in q/o, k/v, lse, and its lse bytes
    if (by_batch) {
      qo = static_cast<size_t>(u0) * Sq * row_b;
      ko = static_cast<size_t>(u0) * Sk * row_b;
      lo = static_cast<size_t>(u0) * H * Sq * 4;
      ls = static_cast<size_t>(nu) * H * Sq * 4;
      const size_t qs = static_cast<size_t>(nu) * Sq * row_b, ks = static_cast<size_t>(nu) * Sk * row_b;
      if ((e = cudaMemcpyAsync(q_d + qo, qh + qo, qs, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess ||
          (e = cudaMemcpyAsync(k_d + ko, kh + ko, ks, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess ||
          (e = cudaMemcpyAsync(v_d + ko, vh + ko, ks, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess) {
        rc = fail_cuda(e, "copy in");
        break;
      }
    } else {
      qo = ko = static_cast<size_t>(u0) * d * 2;
      lo = static_cast<size_t>(u0) * Sq * 4;
      ls = static_cast<size_t>(nu) * Sq * 4;
      const size_t wb = static_cast<size_t>(nu) * d * 2;
      if ((e = cudaMemcpy2DAsync(q_d + qo, row_b, qh + qo, row_b, wb, Sq, cudaMemcpyHostToDevice, hp.in)) !=
              cudaSuccess ||
          (e = cudaMemcpy2DAsync(k_d + ko, row_b, kh + ko, row_b, wb, Sk, cudaMemcpyHostToDevice, hp.in)) !=
              cudaSuccess ||
          (e = cudaMemcpy2DAsync(v_d + ko, row_b, vh + ko, row_b, wb, Sk, cudaMemcpyHostToDevice, hp.in)) !=
              cudaSuccess) {
        rc = fail_cuda(e, "copy in");
        break;
      }
    }
    if ((e = cudaEventRecord(hp.in_done[c], hp.in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, hp.in_done[c], 0)) != cudaSuccess) {
      rc = fail_cuda(e, "order");
      break;
    }
    float* lslice = reinterpret_cast<float*>(l_d + lo);
    if (by_batch) {
      rc = attn_fwd(q_d + qo, k_d + ko, v_d + ko, o_d + qo, lslice, nu, H, Sq, Sk, d, scale, causal, stream);
    } else {
      attn_layout lay;
      std::memset(&lay, 0, sizeof(lay));
      lay.struct_size = sizeof(lay);
      lay.causal_align = ATTN_CAUSAL_TOP_LEFT;
      const long long hd = static_cast<long long>(H) * d;
      for (long long* st : {lay.q_strides, lay.o_strides}) {
        st[0] = Sq * hd;
        st[1] = hd;
        st[2] = d;
      }
      for (long long* st : {lay.k_strides, lay.v_strides}) {
        st[0] = Sk * hd;
        st[1] = hd;
        st[2] = d;
      }
      rc = attn_fwd_layout(q_d + qo, k_d + ko, v_d + ko, o_d + qo, lslice, 1, nu, Sq, Sk, d, scale, causal, &lay,
                           nullptr, stream);
    }
    if (rc != ATTN_OK) break;
    if ((e = cudaEventRecord(hp.k_done[c], stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp.out, hp.k_done[c], 0)) != cudaSuccess) {
      rc = fail_cuda(e, "order");
      break;
    }
    if (by_batch) {
      e = cudaMemcpyAsync(oh + qo, o_d + qo, static_cast<size_t>(nu) * Sq * row_b, cudaMemcpyDeviceToHost, hp.out);
    } else {
      e = cudaMemcpy2DAsync(oh + qo, row_b, o_d + qo, row_b, static_cast<size_t>(nu) * d * 2, Sq,
                            cudaMemcpyDeviceToHost, hp.out);
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(lh + lo, l_d + lo, ls, cudaMemcpyDeviceToHost, hp.out);
    if (e != cudaSuccess) rc = fail_cuda(e, "copy out");
  }
  // Whatever happened, the caller's stream waits for everything enqueued on
  // the internal streams.
  cudaError_t e1 = cudaEventRecord(hp.end, hp.out), e2 = cudaSuccess, e3 = cudaSuccess, e4 = cudaSuccess;
  if (e1 == cudaSuccess) e2 = cudaStreamWaitEvent(stream, hp.end, 0);
  e3 = cudaEventRecord(hp.end, hp.in);  // (the copies in precede the kernels, which precede the copies out)
  if (e3 == cudaSuccess) e4 = cudaStreamWaitEvent(stream, hp.end, 0);
  if (rc == ATTN_OK && (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess))
    rc = fail_cuda(e1 != cudaSuccess ? e1 : e2 != cudaSuccess ? e2 : e3 != cudaSuccess ? e3 : e4, "join");
  return rc;
}

}  // namespace attn

extern "C" {

int attn_version(void) { return 100; }

const char* attn_strerror(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "invalid shape (B, H, Sq, Sk must be >= 1 and the grid must fit)";
    case ATTN_ERR_HEAD_DIM: return "head dim must be 64 or 128";
    case ATTN_ERR_SCALE: return "scale must be finite and > 0";
    case ATTN_ERR_ALIGN: return "device pointers must be 16-byte aligned";
    case ATTN_ERR_ARCH: return "no usable device of compute capability 10.3 (GB300)";
    case ATTN_ERR_LAUNCH: return "CUDA call failed (see attn_last_cuda_error)";
    case ATTN_ERR_TIMEOUT: return "a kernel pipeline wait exceeded its time limit; outputs are invalid";
    case ATTN_ERR_OPTION: return "an attn_options field is out of range";
    case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ATTN_ERR_STATIC_LIMIT: return "problem larger than the static workspace of attn_fwd_host_static";
    case ATTN_ERR_LAYOUT:
      return "invalid attn_layout (H not a multiple of num_kv_heads, a stride not a positive multiple of 8, "
             "or an unknown causal_align)";
    default: return "unknown status";
  }
}

const char* attn_last_cuda_error(void) { return t_last_error; }

int attn_fwd_layout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq, int Sk,
                    int d, float scale, int causal, const attn_layout* layout, const attn_options* opts,
                    cudaStream_t stream) {
  int rc = check_args(q, k, v, o, lse, B, H, Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  int H_kv = H;
  bool bottom_right = false;
  long long qs[3], ks[3], vs[3], os[3];
  {
    static const long long zero[3] = {0, 0, 0};
    const long long* qi = zero;
    const long long* ki = zero;
    const long long* vi = zero;
    const long long* oi = zero;
    if (layout != nullptr) {
      if (layout->struct_size < sizeof(attn_layout)) return ATTN_ERR_LAYOUT;
      if (layout->num_kv_heads < 0) return ATTN_ERR_LAYOUT;
      if (layout->num_kv_heads > 0) H_kv = layout->num_kv_heads;
      if (H % H_kv != 0) return ATTN_ERR_LAYOUT;
      if (layout->causal_align != ATTN_CAUSAL_TOP_LEFT && layout->causal_align != ATTN_CAUSAL_BOTTOM_RIGHT)
        return ATTN_ERR_LAYOUT;
      bottom_right = causal && layout->causal_align == ATTN_CAUSAL_BOTTOM_RIGHT;
      qi = layout->q_strides;
      ki = layout->k_strides;
      vi = layout->v_strides;
      oi = layout->o_strides;
    }
    const long long hd = static_cast<long long>(H) * d, kd = static_cast<long long>(H_kv) * d;
    if (!resolve_strides(qi, Sq * hd, hd, d, qs) || !resolve_strides(ki, Sk * kd, kd, d, ks) ||
        !resolve_strides(vi, Sk * kd, kd, d, vs) || !resolve_strides(oi, Sq * hd, hd, d, os))
      return ATTN_ERR_LAYOUT;
  }
  Opts op;
  if ((rc = parse_options(opts, d, &op)) != ATTN_OK) return rc;
  int dev = -1;
  rc = current_device(&dev);
  if (rc != ATTN_OK) return rc;

  // Causal offset: key j is visible to row i iff j ≤ i + coff.  Bottom-right
  // alignment with Sq > Sk leaves the first Sq − Sk rows without a key: they
  // are written by fill_unseen_rows, and the kernel runs on the remaining
  // rows, a problem with Sq = Sk and offset 0 (every tile then sees a key).
  const int lse_pitch = Sq;
  int coff = bottom_right ? Sk - Sq : 0;
  if (coff < 0) {
    const int unseen = -coff;
    const long long n = static_cast<long long>(B) * H * unseen;
    const int threads = 256;
    const int blocks = static_cast<int>(n / threads + 1 < 4096 ? n / threads + 1 : 4096);
    fill_unseen_rows<<<blocks, threads, 0, stream>>>(static_cast<uint16_t*>(o), os[0], os[1], os[2], lse, lse_pitch,
                                                      B, H, unseen, d);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "row fill launch");
    q = static_cast<const uint16_t*>(q) + static_cast<long long>(unseen) * qs[1];
    o = static_cast<uint16_t*>(o) + static_cast<long long>(unseen) * os[1];
    lse += unseen;
    Sq = Sk;
    coff = 0;
  }

  attn::LaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  if ((rc = encode_bshd(&a.q, q, B, Sq, H, d, qs)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.k, k, B, Sk, H_kv, d, ks)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.v, v, B, Sk, H_kv, d, vs)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.o, o, B, Sq, H, d, os)) != ATTN_OK) return rc;
  const int n_qt = (Sq + 127) / 128;
  a.p.o = o;
  a.p.lse = lse;
  a.p.o_sb = os[0];
  a.p.o_ss = os[1];
  a.p.o_sh = os[2];
  a.p.B = B;
  a.p.H = H;
  a.p.Sq = Sq;
  a.p.Sk = Sk;
  a.p.group = H / H_kv;
  a.p.coff = coff;
  a.p.lse_pitch = lse_pitch;
  a.p.n_qt = n_qt;
  a.p.n_tiles = n_qt * B * H;
  return launch(a, op, dev, d, causal, scale, stream);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int n_seq, int total_q, int total_k, int max_seqlen_q, int H, int H_kv,
                    int d, float scale, int causal, int causal_align, const attn_options* opts, cudaStream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr || cu_seqlens_q == nullptr ||
      cu_seqlens_k == nullptr)
    return ATTN_ERR_NULL;
  if (n_seq < 1 || total_q < 1 || total_k < 1 || max_seqlen_q < 1 || H < 1) return ATTN_ERR_SHAPE;
  const long long n_qt = (static_cast<long long>(max_seqlen_q) + 127) / 128;
  if (static_cast<long long>(n_seq) * H * n_qt > 0x7FFFFFFFLL) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEAD_DIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0 || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u) != 0)
    return ATTN_ERR_ALIGN;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_LAYOUT;
  if (causal_align != ATTN_CAUSAL_TOP_LEFT && causal_align != ATTN_CAUSAL_BOTTOM_RIGHT) return ATTN_ERR_LAYOUT;
  Opts op;
  int rc = parse_options(opts, d, &op);
  if (rc != ATTN_OK) return rc;
  if (op.poly != 0u) return ATTN_ERR_OPTION;  // packed sequences: all-MUFU exp2 only
  int dev = -1;
  if ((rc = current_device(&dev)) != ATTN_OK) return rc;

  // One "batch" of total rows each; the kernel finds each sequence's rows
  // through the offset tables.
  const long long hd = static_cast<long long>(H) * d, kd = static_cast<long long>(H_kv) * d;
  const long long qs[3] = {total_q * hd, hd, d}, ks[3] = {total_k * kd, kd, d};
  attn::LaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  if ((rc = encode_bshd(&a.q, q, 1, total_q, H, d, qs)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.k, k, 1, total_k, H_kv, d, ks)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.v, v, 1, total_k, H_kv, d, ks)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.o, o, 1, total_q, H, d, qs)) != ATTN_OK) return rc;
  a.p.o = o;
  a.p.lse = lse;
  a.p.o_sb = qs[0];
  a.p.o_ss = qs[1];
  a.p.o_sh = qs[2];
  a.p.B = n_seq;
  a.p.H = H;
  a.p.Sq = max_seqlen_q;
  a.p.Sk = 0;
  a.p.group = H / H_kv;
  a.p.coff = 0;
  a.p.lse_pitch = total_q;
  a.p.cu_q = cu_seqlens_q;
  a.p.cu_k = cu_seqlens_k;
  a.p.total_q = total_q;
  a.p.total_k = total_k;
  a.p.bottom_right = (causal && causal_align == ATTN_CAUSAL_BOTTOM_RIGHT) ? 1 : 0;
  a.p.n_qt = static_cast<int>(n_qt);
  a.p.n_tiles = static_cast<int>(n_qt * n_seq * H);
  return launch(a, op, dev, d, causal, scale, stream);
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq, int Sk, int d,
                float scale, int causal, const attn_options* opts, cudaStream_t stream) {
  return attn_fwd_layout(q, k, v, o, lse, B, H, Sq, Sk, d, scale, causal, nullptr, opts, stream);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq, int Sk, int d,
             float scale, int causal, cudaStream_t stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, Sq, Sk, d, scale, causal, nullptr, stream);
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, void* o, float* lse, int B, int H, int Sq, int Sk,
                 int d, float scale, float descale_q, float descale_k, float descale_v, int causal,
                 cudaStream_t stream) {
  return attn_fwd_fp8_ex(q8, k8, v8, o, lse, B, H, Sq, Sk, d, scale, descale_q, descale_k, descale_v, causal,
                         nullptr, stream);
}

int attn_fwd_fp8_ex(const void* q8, const void* k8, const void* v8, void* o, float* lse, int B, int H, int Sq,
                    int Sk, int d, float scale, float descale_q, float descale_k, float descale_v, int causal,
                    const attn_options* opts, cudaStream_t stream) {
  if (q8 == nullptr || k8 == nullptr || v8 == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_SHAPE;
  const long long n_qt = (static_cast<long long>(Sq) + 127) / 128;
  if (static_cast<long long>(B) * H * n_qt > 0x7FFFFFFFLL) return ATTN_ERR_SHAPE;
  if (d != 128) return ATTN_ERR_HEAD_DIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  for (float f : {descale_q, descale_k, descale_v})
    if (!std::isfinite(f) || !(f > 0.f)) return ATTN_ERR_SCALE;
  const float sl = scale * descale_q * descale_k * 1.4426950408889634f;
  if (!std::isfinite(sl) || !(sl > 0.f)) return ATTN_ERR_SCALE;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  Opts op;
  int rc = parse_options(opts, d, &op);
  if (rc != ATTN_OK) return rc;
  if (opts != nullptr && (opts->rescale_threshold != 0.f || opts->poly_exp2_mask != 0u || opts->counters != nullptr))
    return ATTN_ERR_OPTION;
  int dev = -1;
  rc = current_device(&dev);
  if (rc != ATTN_OK) return rc;
  attn::LaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  const long long hd = static_cast<long long>(H) * d;
  const long long os[3] = {Sq * hd, hd, d};
  if ((rc = encode_bshd_u8(&a.q, q8, B, Sq, H, d)) != ATTN_OK) return rc;
  if ((rc = encode_bshd_u8(&a.k, k8, B, Sk, H, d)) != ATTN_OK) return rc;
  if ((rc = encode_bshd_u8(&a.v, v8, B, Sk, H, d)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.o, o, B, Sq, H, d, os)) != ATTN_OK) return rc;
  a.p.o = o;
  a.p.lse = lse;
  a.p.o_sb = os[0];
  a.p.o_ss = os[1];
  a.p.o_sh = os[2];
  a.p.B = B;
  a.p.H = H;
  a.p.Sq = Sq;
  a.p.Sk = Sk;
  a.p.group = 1;
  a.p.coff = 0;
  a.p.lse_pitch = Sq;
  a.p.n_qt = static_cast<int>(n_qt);
  a.p.n_tiles = static_cast<int>(n_qt * B * H);
  a.p.status = g_dev[dev].status;
  a.p.scale_log2 = sl;
  a.p.o_scale = descale_v / 448.0f;
  a.p.timeout_ns = static_cast<uint64_t>(op.timeout_ms) * 1000000ull;
  a.p.test_flags = op.test_flags;
  a.grid = a.p.n_tiles < g_dev[dev].sms ? a.p.n_tiles : g_dev[dev].sms;
  a.sms = g_dev[dev].sms;
  a.device = dev;
  a.stream = stream;
  const cudaError_t e = attn::launch_fwd_fp8(a, causal != 0);
  if (e != cudaSuccess) return fail_cuda(e, "FP8 attention kernel launch");
  return ATTN_OK;
}

namespace {
// Workspace: −LSE·log2 e and D per query row ([B·H, pitch] each), then the
// one-pass kernel's fp32 dQ accumulator [B·H, pitch, 64] (it runs at d = 64).
size_t bwd_vec_bytes(int B, int H, int Sq) {
  const size_t pitch = (static_cast<size_t>(Sq) + 127) / 128 * 128;
  return (2 * static_cast<size_t>(B) * H * pitch * 4 + 255) & ~static_cast<size_t>(255);
}

// 2-D map over the fp32 accumulator: d values per row, B·H·pitch rows; box
// 32 values × 32 rows (one 128-byte swizzle row per row).
int encode_dq_acc(CUtensorMap* m, float* acc, long long rows, int d) {
  auto enc = get_encode_fn();
  if (enc == nullptr) {
    std::snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled unavailable");
    return ATTN_ERR_LAUNCH;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, acc, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled failed (CUresult %d)",
                  static_cast<int>(r));
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}
}  // namespace

size_t attn_bwd_workspace_size(int B, int H, int Sq) {
  if (B < 1 || H < 1 || Sq < 1) return 0;
  const size_t pitch = (static_cast<size_t>(Sq) + 127) / 128 * 128;
  return bwd_vec_bytes(B, H, Sq) + static_cast<size_t>(B) * H * pitch * 64 * 4;
}

int attn_bwd_layout(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int d, float scale, int causal,
                    const attn_layout* layout, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return attn_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, B, H, Sq, Sk, d, scale, causal, layout, 0u, workspace,
                     workspace_bytes, stream);
}

int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int d, float scale, int causal,
                const attn_layout* layout, unsigned int flags, void* workspace, size_t workspace_bytes,
                cudaStream_t stream) {
  int rc = check_args(q, k, v, o, lse, B, H, Sq, Sk, d, scale);
  if (rc != ATTN_OK) return rc;
  if ((flags & ~static_cast<unsigned int>(ATTN_BWD_DETERMINISTIC)) != 0) return ATTN_ERR_OPTION;
  int H_kv = H;
  bool bottom_right = false;
  static const long long zero3[3] = {0, 0, 0};
  const long long *qi = zero3, *ki = zero3, *vi = zero3, *oi = zero3;
  if (layout != nullptr) {
    if (layout->struct_size < sizeof(attn_layout) || layout->num_kv_heads < 0) return ATTN_ERR_LAYOUT;
    if (layout->num_kv_heads > 0) H_kv = layout->num_kv_heads;
    if (H % H_kv != 0) return ATTN_ERR_LAYOUT;
    if (layout->causal_align != ATTN_CAUSAL_TOP_LEFT && layout->causal_align != ATTN_CAUSAL_BOTTOM_RIGHT)
      return ATTN_ERR_LAYOUT;
    bottom_right = causal && layout->causal_align == ATTN_CAUSAL_BOTTOM_RIGHT;
    qi = layout->q_strides;
    ki = layout->k_strides;
    vi = layout->v_strides;
    oi = layout->o_strides;
  }
  // q, k, v and o may be strided (the layout's strides); dout, dq, dk, dv are dense.
  const long long hd = static_cast<long long>(H) * d, kd = static_cast<long long>(H_kv) * d;
  long long qs[3], ks[3], vs[3], os[3];
  if (!resolve_strides(qi, Sq * hd, hd, d, qs) || !resolve_strides(ki, Sk * kd, kd, d, ks) ||
      !resolve_strides(vi, Sk * kd, kd, d, vs) || !resolve_strides(oi, Sq * hd, hd, d, os))
    return ATTN_ERR_LAYOUT;
  const long long qd_[3] = {Sq * hd, hd, d}, kd_[3] = {Sk * kd, kd, d};  // dense dout, dq and dk, dv
  if (dout == nullptr || dq == nullptr || dk == nullptr || dv == nullptr) return ATTN_ERR_NULL;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv)) return ATTN_ERR_ALIGN;
  const long long n_kt = (static_cast<long long>(Sk) + 127) / 128;
  if (static_cast<long long>(B) * H_kv * n_kt > 0x7FFFFFFFLL) return ATTN_ERR_SHAPE;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < attn_bwd_workspace_size(B, H, Sq))
    return ATTN_ERR_WORKSPACE;
  int dev = -1;
  if ((rc = current_device(&dev)) != ATTN_OK) return rc;

  const int pitch = (Sq + 127) / 128 * 128;
  float* lse2 = static_cast<float*>(workspace);
  float* dvec = lse2 + static_cast<size_t>(B) * H * pitch;
  // At d = 64 one pass (dQ added up in fp32 across key tiles, in an order
  // that varies between runs) unless the caller asks for bit-reproducible
  // gradients; at d = 128 the two passes (faster there: the one-pass
  // kernel's dQ reduce-adds are bound by the L2's reduction rate).  The
  // kernel addresses accumulator rows with 32-bit coordinates.
  const long long acc_rows = static_cast<long long>(B) * H * pitch;
  const bool fused = (flags & ATTN_BWD_DETERMINISTIC) == 0 && d == 64 && acc_rows <= 0x7FFFFFFFLL;
  float* dq_acc = fused ? reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_vec_bytes(B, H, Sq)) : nullptr;
  cudaError_t e = attn::launch_bwd_prep(o, os, dout, lse, lse2, dvec, dq_acc, B, H, Sq, pitch, d, stream);
  if (e != cudaSuccess) return fail_cuda(e, "backward preparation launch");

  attn::BwdLaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  a.p.lse2 = lse2;
  a.p.dvec = dvec;
  a.p.status = g_dev[dev].status;
  a.p.B = B;
  a.p.H = H;
  a.p.Sq = Sq;
  a.p.Sk = Sk;
  a.p.pitch = pitch;
  a.p.coff = bottom_right ? Sk - Sq : 0;  // negative: rows without keys, whose gradients are zero
  a.p.group = H / H_kv;
  a.p.scale_log2 = scale * 1.4426950408889634f;
  a.p.scale = scale;
  a.p.timeout_ns = static_cast<uint64_t>(kDefaultTimeoutMs) * 1000000ull;
  a.causal = causal != 0;
  a.device = dev;
  a.stream = stream;
  // dK, dV: rows are keys; the queries' Q and dO stream past them.
  if ((rc = encode_bshd(&a.x, k, B, Sk, H_kv, d, ks)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.x2, v, B, Sk, H_kv, d, vs)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.a, q, B, Sq, H, d, qs)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.b, dout, B, Sq, H, d, qd_)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.o0, dv, B, Sk, H_kv, d, kd_)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.o1, dk, B, Sk, H_kv, d, kd_)) != ATTN_OK) return rc;
  a.p.n_rt = static_cast<int>(n_kt);
  a.grid = static_cast<int>(n_kt * B * H_kv);
  if (fused) {
    if ((rc = encode_dq_acc(&a.dq, dq_acc, acc_rows, d)) != ATTN_OK) return rc;
    a.mode = 2;
    if ((e = attn::launch_bwd(a, d)) != cudaSuccess) return fail_cuda(e, "backward fused launch");
    e = attn::launch_bwd_dq_convert(dq_acc, dq, B, H, Sq, pitch, d, scale, g_dev[dev].sms, stream);
    if (e != cudaSuccess) return fail_cuda(e, "backward dQ conversion launch");
    return ATTN_OK;
  }
  a.dq = a.o0;  // unused by the two-pass kernels
  a.mode = 1;
  if ((e = attn::launch_bwd(a, d)) != cudaSuccess) return fail_cuda(e, "backward dK/dV launch");
  // dQ: rows are queries; K and V stream past them.
  if ((rc = encode_bshd(&a.x, q, B, Sq, H, d, qs)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.x2, dout, B, Sq, H, d, qd_)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.a, k, B, Sk, H_kv, d, ks)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.b, v, B, Sk, H_kv, d, vs)) != ATTN_OK) return rc;
  if ((rc = encode_bshd(&a.o0, dq, B, Sq, H, d, qd_)) != ATTN_OK) return rc;
  a.o1 = a.o0;  // unused by the dQ pass
  a.p.n_rt = (Sq + 127) / 128;
  a.grid = a.p.n_rt * B * H;
  a.mode = 0;
  if ((e = attn::launch_bwd(a, d)) != cudaSuccess) return fail_cuda(e, "backward dQ launch");
  return ATTN_OK;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, int B, int H, int Sq, int Sk, int d, float scale, int causal, void* workspace,
             size_t workspace_bytes, cudaStream_t stream) {
  return attn_bwd_layout(q, k, v, o, lse, dout, dq, dk, dv, B, H, Sq, Sk, d, scale, causal, nullptr, workspace,
                         workspace_bytes, stream);
}

size_t attn_fwd_host_workspace_size(int B, int H, int Sq, int Sk, int d) {
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1 || (d != 64 && d != 128)) return 0;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t qo = up(static_cast<size_t>(B) * Sq * H * d * 2);
  const size_t kv = up(static_cast<size_t>(B) * Sk * H * d * 2);
  const size_t ls = up(static_cast<size_t>(B) * H * Sq * 4);
  return 2 * qo + 2 * kv + ls;
}

int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h, int B, int H, int Sq,
                  int Sk, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream) {
  return attn::fwd_host(q_h, k_h, v_h, o_h, lse_h, B, H, Sq, Sk, d, scale, causal, workspace, workspace_bytes,
                        stream, true);
}

int attn_get_status(cudaStream_t stream) {
  int dev = -1;
  int rc = current_device(&dev);
  if (rc != ATTN_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  unsigned int v = 0;
  if ((e = cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(v))) != cudaSuccess)
    return fail_cuda(e, "read status");
  if (v != 0) {
    const unsigned int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero))) != cudaSuccess)
      return fail_cuda(e, "clear status");
    return ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

}  // extern "C"

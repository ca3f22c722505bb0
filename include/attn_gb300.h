/*
 * attn_gb300.h — C ABI of the exact attention forward library (GB300, sm_103a).
 *
 * The operation (every entry point below computes it):
 *   O = softmax(scale · Q Kᵀ) V, optionally causal, and the per-row
 *   log-sum-exp LSE.  Scaled attention softmax(QKᵀ/√d)V is defined in
 *   "FlashAttention-4 no Blackwell B200 …", section "Por que o Blackwell exige
 *   mais do que multiplicações rápidas"; the call shape (q, k, v, softmax_scale,
 *   causal) and the (batch, seq, heads, head_dim) layout follow the Python call
 *   in "FlashAttention-3: Pipeline Assíncrono …", section "Implementando
 *   FlashAttention-3 em produção".  The kernels compute it tile by tile with
 *   an online softmax ("FlashAttention 4: Atenção Mais Rápida …", section
 *   "Novidades no FlashAttention 4"), so the Sq×Sk score matrix never reaches
 *   device memory; the result equals the plain definition up to rounding.
 *
 * Definitions (per batch b, head h, query row i):
 *   s_ij   = scale · Σ_c q[b,i,h,c] · k[b,j,h,c]
 *   V_i    = { j : 0 ≤ j < Sk, and j ≤ i when causal }   (top-left alignment)
 *   LSE_i  = ln Σ_{j∈V_i} exp(s_ij)                        (natural log)
 *   O_i    = Σ_{j∈V_i} exp(s_ij − LSE_i) · v[b,j,h,:]
 *   A row with no visible key (possible only when causal and Sk = 0, which the
 *   shape checks reject) would get O = 0 and LSE = −inf.
 *
 * Layouts (all dense, row-major, no padding):
 *   q   bf16  [B, Sq, H, d]      k, v  bf16  [B, Sk, H, d]
 *   o   bf16  [B, Sq, H, d]      lse   fp32  [B, H, Sq]
 * Arithmetic: bf16 inputs, fp32 accumulation in tensor memory, fp32 softmax,
 * probabilities rounded to bf16 for the P·V product, row sums accumulated in
 * fp32 from unrounded probabilities, O rounded once to bf16 (RNE).
 *
 * Ownership: the caller owns every buffer; the library allocates nothing per
 * call and frees nothing.  The library keeps one 4-byte status word per
 * device in a statically sized device variable.
 *
 * Asynchrony and errors: every launching call is asynchronous on `stream`
 * (0 = the legacy default stream) and returns after the launch.  A negative
 * return code means the call was rejected BEFORE any launch and nothing was
 * written.  Device-side failures (a pipeline wait that exceeded its time
 * limit) are reported later by attn_get_status().
 *
 * Requirements: compute capability 10.3 (GB300); d ∈ {64, 128}; device
 * pointers 16-byte aligned (TMA requirement; 128-byte alignment is faster,
 * and PyTorch's allocator gives 256 bytes); B, H, Sq, Sk ≥ 1.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  0 = success; negative = rejected or failed. */
enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = -1,      /* a required pointer is NULL */
  ATTN_ERR_SHAPE = -2,     /* B, H, Sq or Sk < 1, or a size overflows the kernel's index range */
  ATTN_ERR_HEAD_DIM = -3,  /* d is not 64 or 128 */
  ATTN_ERR_SCALE = -4,     /* scale is not finite or not > 0 */
  ATTN_ERR_ALIGN = -5,     /* a device pointer is not 16-byte aligned */
  ATTN_ERR_ARCH = -6,      /* no device, or the current device is not compute capability 10.3 */
  ATTN_ERR_LAUNCH = -7,    /* a CUDA call failed; attn_last_cuda_error() has the message */
  ATTN_ERR_TIMEOUT = -8,   /* (attn_get_status) a kernel wait exceeded its limit; outputs invalid */
  ATTN_ERR_OPTION = -9,    /* an attn_options field is out of range */
  ATTN_ERR_WORKSPACE = -10, /* workspace missing, misaligned or smaller than required */
  ATTN_ERR_STATIC_LIMIT = -11, /* problem needs more than ATTN_STATIC_WORKSPACE_BYTES (attn_fwd_host_static) */
  ATTN_ERR_LAYOUT = -12       /* an attn_layout field is invalid (head grouping, strides, causal alignment) */
};

/*
 * attn_fwd — exact attention forward on device buffers.
 *   q, k, v : device, bf16, layouts above (read only).
 *   o       : device, bf16 [B, Sq, H, d] (written).
 *   lse     : device, fp32 [B, H, Sq] (written).
 *   B, H    : batch size and number of heads (K/V have the same H).
 *   Sq, Sk  : query and key sequence lengths (may differ; any value ≥ 1).
 *   d       : head dimension, 64 or 128.
 *   scale   : multiplier of QKᵀ (the pages pass 1/√d), finite and > 0.
 *   causal  : 0 = full attention; non-zero = key j visible to query i iff j ≤ i.
 *   stream  : CUDA stream of the caller's context.
 * Returns ATTN_OK after launching, or a negative code without launching.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int Sq, int Sk, int d, float scale, int causal,
             cudaStream_t stream);

/*
 * Tuning and diagnostic options for attn_fwd_ex().  Zero-initialise and set
 * struct_size = sizeof(attn_options); a zero field means "default".
 *
 * rescale_threshold — τ of the conditional online rescaling ("FlashAttention 4:
 *   Atenção Mais Rápida …", section "Reescalonamento Softmax Online Mais
 *   Inteligente"): a row's running maximum (log2 domain) is only replaced when
 *   a new block's maximum exceeds it by more than τ; otherwise probabilities
 *   up to 2^τ are accumulated against the stale maximum.  The result does not
 *   depend on τ beyond rounding.  Range [0, 64]; a negative value selects
 *   τ = 0 (rescale on every increase); 0 selects the default 32.
 * poly_exp2_mask — which 16-column chunks of each 128-key block compute exp2
 *   with the FMA-pipe cubic polynomial instead of the MUFU unit ("…", section
 *   "Exponenciais de Software via Núcleos CUDA").  Bit c (0..7) selects chunk
 *   c.  The splits compiled in are 0x01 (1/8), 0x11 (1/4), 0x55 (1/2) and
 *   0xFF (all); 0x100 selects none (all MUFU); 0 selects the default for the
 *   head dim; any other value is rejected with ATTN_ERR_OPTION.
 * counters — optional device pointer to 2 zero-initialised uint64 values; when
 *   non-NULL the kernel adds the number of rescales to counters[0] and the
 *   number of (row, block) softmax updates to counters[1].  A rescale is
 *   counted per row, key block and running maximum: at d = 128 each 128-key
 *   block is processed as two 64-key halves with running maxima of their own;
 *   at d = 64 a row keeps one running maximum (two halves under
 *   ATTN_TEST_FALLBACK_KERNEL).
 * timeout_ms — time limit of every pipeline wait inside the kernel (default
 *   4000 ms); on expiry the kernel stops, leaves outputs invalid and flags
 *   ATTN_ERR_TIMEOUT for attn_get_status().  The limit is measured in wall
 *   time (the GPU's global timer): on a GPU time-sliced between processes,
 *   time spent while this context is switched out counts too, so a very long
 *   call on a heavily shared GPU can report ATTN_ERR_TIMEOUT without any
 *   fault; raise the limit there.
 * test_flags — for tests only; 0 in normal use.
 *   ATTN_TEST_WITHHOLD_KV: the loader never issues the K/V copies, so the
 *   MMA issuer's first wait cannot complete and must run into timeout_ms; the
 *   kernel then stops cleanly (no fault, TMEM released) and attn_get_status()
 *   returns ATTN_ERR_TIMEOUT.  Outputs are not written.
 *   ATTN_TEST_FALLBACK_KERNEL: at d = 64 (bf16) and for FP8 inputs, run the
 *   kernel that serves when the full-row kernel (two CTAs per SM) is not
 *   compiled to the register count its register split needs — the
 *   two-warpgroup kernel of d = 128, or the one-CTA FP8 kernel — so that this
 *   fallback can be tested.  Same results within the tolerances.
 */
#define ATTN_TEST_WITHHOLD_KV 1u
#define ATTN_TEST_FALLBACK_KERNEL 2u
typedef struct attn_options {
  size_t struct_size;
  float rescale_threshold;
  unsigned int poly_exp2_mask;
  unsigned long long* counters;
  unsigned int timeout_ms;
  unsigned int test_flags;
} attn_options;

/* attn_fwd with options (opts may be NULL: same as attn_fwd). */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int Sq, int Sk, int d, float scale, int causal,
                const attn_options* opts, cudaStream_t stream);

/*
 * Layout and head grouping for attn_fwd_layout().  Zero-initialise and set
 * struct_size = sizeof(attn_layout); a zero field keeps attn_fwd's default.
 *
 * num_kv_heads — H_kv, the number of key/value heads.  Grouped-query attention
 *   ("FlashAttention 4: Atenção Mais Rápida …", section "Compatibilidade e
 *   status atual": several query heads share one key/value projection): H must
 *   be a multiple of H_kv and query head h reads key/value head h / (H / H_kv);
 *   k and v are then [B, Sk, H_kv, d].  0 selects H (multi-head attention);
 *   1 is multi-query attention.
 * causal_align — used when causal != 0.  ATTN_CAUSAL_TOP_LEFT (0, the
 *   default and attn_fwd's rule): key j is visible to query i iff j ≤ i.
 *   ATTN_CAUSAL_BOTTOM_RIGHT (1): iff j ≤ i + Sk − Sq, so the last query row
 *   sees every key.  Rows that see no key (bottom-right with Sq > Sk: the
 *   first Sq − Sk rows) get O = 0 and LSE = −inf.  The pages fix no rule for
 *   Sq ≠ Sk; both common ones are offered.
 * q_strides, k_strides, v_strides, o_strides — element strides of the batch,
 *   sequence and head dimensions of each tensor; the d elements of one head
 *   row stay contiguous.  All three zero selects the dense layout above.
 *   Otherwise each must be a positive multiple of 8 elements (16 bytes, a TMA
 *   requirement) below 2^38.  Example: a packed [B, S, 3, H, d] QKV tensor
 *   gives q, k, v at element offsets 0, H·d, 2·H·d with strides
 *   (3·S·H·d, 3·H·d, d).  o must not overlap q, k, v or lse.
 * LSE stays dense [B, H, Sq].
 */
#define ATTN_CAUSAL_TOP_LEFT 0
#define ATTN_CAUSAL_BOTTOM_RIGHT 1
typedef struct attn_layout {
  size_t struct_size;
  int num_kv_heads;
  int causal_align;
  long long q_strides[3];
  long long k_strides[3];
  long long v_strides[3];
  long long o_strides[3];
} attn_layout;

/*
 * attn_fwd_layout — attn_fwd_ex with a layout (layout may be NULL: dense
 * multi-head tensors, top-left causal alignment, the same as attn_fwd_ex).
 * Argument meanings, ownership and asynchrony as attn_fwd; additional errors:
 * ATTN_ERR_LAYOUT for an invalid layout.  When rows see no key, their O and
 * LSE are written by a second, small kernel on the same stream.
 */
int attn_fwd_layout(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int Sq, int Sk, int d, float scale, int causal,
                    const attn_layout* layout, const attn_options* opts, cudaStream_t stream);

/*
 * attn_fwd_varlen — attention over a batch of sequences of different lengths
 * packed along the rows ("FlashAttention 4: …", section "Compatibilidade e
 * status atual", names variable-length batches, processed without padding).
 *   q, o          : device, bf16 [total_q, H, d] (dense); o is written.
 *   k, v          : device, bf16 [total_k, H_kv, d] (dense).
 *   lse           : device, fp32 [H, total_q] (written).
 *   cu_seqlens_q  : device, int32 [n_seq + 1], ascending, cu_seqlens_q[0] = 0,
 *                   cu_seqlens_q[n_seq] = total_q: sequence s owns query rows
 *                   [cu_seqlens_q[s], cu_seqlens_q[s+1]).
 *   cu_seqlens_k  : the same for key/value rows (total_k); sequence s attends
 *                   only to its own keys.  Lengths may be 0.
 *   max_seqlen_q  : host, at least the longest query sequence (it sizes the
 *                   grid; rows of a longer sequence beyond it are not written).
 *   H, H_kv, d, scale : as attn_fwd / attn_layout (H a multiple of H_kv).
 *   causal, causal_align : as attn_fwd / attn_layout, per sequence: with
 *                   bottom-right alignment key j is visible to row i of a
 *                   sequence iff j ≤ i + len_k − len_q.  Rows that see no key
 *                   (also every row of a sequence without keys) get O = 0,
 *                   LSE = −inf.
 * The offset tables are read on the device; offsets outside [0, total] are
 * clamped, so a malformed table gives wrong results but no access outside the
 * tensors.  Returns ATTN_OK after launching, or a negative code (before any
 * launch): ATTN_ERR_NULL, ATTN_ERR_SHAPE (n_seq, total_q, total_k,
 * max_seqlen_q < 1 or the grid does not fit), ATTN_ERR_HEAD_DIM,
 * ATTN_ERR_SCALE, ATTN_ERR_ALIGN (tensors 16-byte, tables 4-byte aligned),
 * ATTN_ERR_LAYOUT (H_kv, causal_align), ATTN_ERR_OPTION (also for a
 * poly_exp2_mask other than the default: this call computes every exp2 on
 * the MUFU unit).
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seq,
                    int total_q, int total_k, int max_seqlen_q,
                    int H, int H_kv, int d, float scale, int causal, int causal_align,
                    const attn_options* opts, cudaStream_t stream);

/*
 * attn_bwd — gradients of attn_fwd's O with respect to q, k and v.
 *   The pages give no backward formulas ("FlashAttention-4 no Blackwell B200
 *   …", section "Redução de tráfego no backward", only says FA4 keeps the
 *   backward's intermediates in tensor memory); this is the derivative of the
 *   definition above for a loss whose gradient with respect to O is dout (the
 *   LSE output is not differentiated).  With P_ij = exp(s_ij − LSE_i) over
 *   visible keys:  dV = Pᵀ·dout,  dP = dout·Vᵀ,  D_i = Σ_c dout_ic·o_ic,
 *   dS = P ∘ (dP − D),  dQ = scale·dS·K,  dK = scale·dSᵀ·Q.
 *   q, k, v, o, dout : device, bf16, dense, layouts as attn_fwd (o and lse as
 *                      attn_fwd returned them for the same q, k, v, scale,
 *                      causal).  Read only.
 *   dq, dk, dv       : device, bf16, shaped like q, k, v (written).
 *   B, H, Sq, Sk, d, scale, causal : as attn_fwd (top-left causal alignment;
 *                      K and V have H heads).
 *   workspace        : caller-owned DEVICE buffer of at least
 *                      attn_bwd_workspace_size(B, H, Sq) bytes, 256-byte
 *                      aligned (holds D and LSE·log2 e per query row and,
 *                      for the one-pass schedule, an fp32 dQ accumulator of
 *                      B·H·⌈Sq/128⌉·128 rows × 64 values; its contents on
 *                      entry do not matter).
 * Arithmetic: bf16 operands, fp32 accumulation in tensor memory, P and dS
 * rounded to bf16 for the products, outputs rounded once to bf16.
 * Schedules.  d = 64 (default): one pass over the key tiles — each key
 * tile's CTA forms S, dP, P and dS once per (query, key) pair, accumulates dK
 * and dV in tensor memory and adds its contribution to dQ into the fp32
 * accumulator in device memory (reduce-add copies); a last kernel scales and
 * rounds dQ.  The fp32 additions into dQ happen in an order that varies from
 * run to run, so dQ can differ in its last bits between runs (dK and dV do
 * not).  d = 128, or attn_bwd_ex() with ATTN_BWD_DETERMINISTIC: two passes
 * (dK/dV, then dQ, which recomputes S and dP), bit-reproducible.
 * Enqueues three kernels on `stream` (D and LSE·log2 e, the pass, the dQ
 * rounding; or D and LSE·log2 e, dK/dV, dQ) and returns; errors as attn_fwd,
 * plus ATTN_ERR_WORKSPACE.
 */
size_t attn_bwd_workspace_size(int B, int H, int Sq);
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int d, float scale, int causal,
             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_bwd_layout — attn_bwd with grouped key/value heads and the causal
 * alignment of an attn_layout (layout may be NULL: the same as attn_bwd).
 * k, v, dk, dv then have num_kv_heads heads: the gradient of a key/value
 * head sums the contributions of every query head of its group.  Rows that
 * see no key (bottom-right with Sq > Sk) get zero dQ.  q, k, v and o may be
 * strided views as attn_layout describes (e.g. slices of a packed QKV
 * tensor; same rules, else ATTN_ERR_LAYOUT); dout, dq, dk and dv are dense
 * [B, S, H(_kv), d].
 */
int attn_bwd_layout(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int d, float scale, int causal,
                    const attn_layout* layout, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_bwd_ex — attn_bwd_layout with schedule flags (0: the same call).
 *   ATTN_BWD_DETERMINISTIC: the two-pass schedule at every head dim; dQ, dK
 *   and dV are then identical bit for bit from run to run.  Results of the
 *   two schedules agree within rounding.
 * Other flag bits: ATTN_ERR_OPTION.  The same workspace rule as attn_bwd.
 */
#define ATTN_BWD_DETERMINISTIC 1u
int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int d, float scale, int causal,
                const attn_layout* layout, unsigned int flags, void* workspace, size_t workspace_bytes,
                cudaStream_t stream);

/*
 * attn_fwd_host — the same operation on HOST buffers, end to end.
 *   q_h, k_h, v_h : host bf16 inputs (layouts above); o_h, lse_h : host outputs.
 *   workspace     : caller-owned DEVICE buffer of at least
 *                   attn_fwd_host_workspace_size(B, H, Sq, Sk, d) bytes,
 *                   256-byte aligned; it holds device copies of q, k, v, o, lse.
 * The problem is cut into up to four slices (of the batch, or of the heads
 * when B = 1 and Sq is a multiple of 4, whose rows are then copied as strided
 * 2-D copies; otherwise it runs as one slice on `stream`); each slice's
 * host→device copies run on a library-owned stream, its kernel on `stream`
 * and its device→host copies on a second library-owned stream, ordered by
 * events, so one slice's copies overlap the others' compute and copies.  The
 * library creates these two streams and their events on a device's first
 * call and keeps them; enqueueing is serialised per device by a mutex.
 * `stream` waits for every copy before any later work on it runs, and the
 * first copy waits for earlier work on `stream`.  The call returns after
 * enqueueing; synchronise `stream` before reading o_h / lse_h.  Host buffers
 * should be page-locked for the copies to be asynchronous.  Argument errors
 * are returned before anything is enqueued.
 */
size_t attn_fwd_host_workspace_size(int B, int H, int Sq, int Sk, int d);
int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                  int B, int H, int Sq, int Sk, int d, float scale, int causal,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_fwd_host_static — attn_fwd_host for callers that cannot allocate device
 * memory.  The pages have no counterpart to this call; it exists for
 * integration.  Some host programs may not call cudaMalloc at all: plugins
 * whose framework owns every byte of device memory through its own allocator
 * (an extra cudaMalloc bypasses its accounting and can fail once the pool has
 * reserved the device), and latency-critical or certified code paths that
 * forbid allocation after start-up (cudaMalloc may synchronise the device).
 * Such callers pass host inputs and outputs only; the device staging area is
 * a fixed array of ATTN_STATIC_WORKSPACE_BYTES (32 MiB) inside this library,
 * which every GPU that loads the library keeps until the process exits.
 *   Arguments and layouts as attn_fwd_host, without the workspace.  Everything
 *   runs on `stream` in one slice (no library streams or events are created).
 *   Problems whose attn_fwd_host_workspace_size() exceeds
 *   ATTN_STATIC_WORKSPACE_BYTES are rejected with ATTN_ERR_STATIC_LIMIT
 *   before anything is enqueued.
 *   Every call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress), which allocates nothing once the array exists.
 *   When the array comes into existence depends on CUDA's module loading:
 *   with lazy loading (the default) the first call on each device loads this
 *   part of the library and reserves the 32 MiB then; with eager loading
 *   (CUDA_MODULE_LOADING=EAGER) loading the library reserves it on every
 *   device.  That reservation is a device allocation and can fail with out
 *   of memory (ATTN_ERR_LAUNCH; attn_last_cuda_error() has the CUDA error)
 *   once another allocator has taken the device, so make one call on each
 *   device at start-up, before pools reserve the device and before any
 *   stream capture.  Later calls allocate nothing.
 *   All calls share the one array, which keeps the last call's contents:
 *   calls whose GPU work overlaps (different streams without ordering, or
 *   several host threads) race on it and must be serialised by the caller.
 *   Nothing in the array needs to start at zero.
 * Enqueues the same copies and kernel as attn_fwd_host; returns after
 * enqueueing, synchronise `stream` before reading o_h / lse_h.
 */
#define ATTN_STATIC_WORKSPACE_BYTES (32u << 20)
int attn_fwd_host_static(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                         int B, int H, int Sq, int Sk, int d, float scale, int causal,
                         cudaStream_t stream);

/*
 * attn_fwd_fp8 — exact attention forward on FP8 (E4M3) inputs.
 *   "FlashAttention-3: Pipeline Assíncrono …", section "Estabilidade em FP8":
 *   two passes over each query tile's keys — the exact row maximum of the
 *   scaled logits first (products accumulated in fp32), then p ≤ 1 and O =
 *   P·V with P rounded to E4M3 under a static scale (448 p).
 *   q8, k8, v8 : device, E4M3 bytes (1 sign, 4 exponent, 3 mantissa bits),
 *                dense [B, Sq, H, d] / [B, Sk, H, d] (read only); they stand
 *                for descale_q·q8, descale_k·k8, descale_v·v8.
 *   o          : device, bf16 [B, Sq, H, d] (written); lse: fp32 [B, H, Sq],
 *                natural log of Σ_visible exp(scale · q_i · k_j) over the
 *                dequantized values.
 *   d          : 128 only (ATTN_ERR_HEAD_DIM otherwise).
 *   scale, descale_q, descale_k, descale_v : finite and > 0 (ATTN_ERR_SCALE).
 *   causal     : top-left alignment (key j visible to row i iff j ≤ i).
 *   Accuracy: O differs from the exact result over the dequantized inputs by
 *   at most Σ_j |p̂_ij − p_ij|·|v_j| / Σ_j p_ij (+ the bf16 rounding of O),
 *   p̂ being p rounded to E4M3 (relative 2^-4, or 2^-10/448 below E4M3's
 *   normal range); LSE is as accurate as the bf16 path's.
 *   Asynchronous on `stream`; errors as attn_fwd.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                 int B, int H, int Sq, int Sk, int d, float scale,
                 float descale_q, float descale_k, float descale_v, int causal,
                 cudaStream_t stream);

/* attn_fwd_fp8 with options (opts may be NULL: same as attn_fwd_fp8).  Only
 * timeout_ms and test_flags apply; rescale_threshold, poly_exp2_mask and
 * counters must be zero (ATTN_ERR_OPTION otherwise): there is no rescaling,
 * the maximum being exact, and every exponential is on the MUFU unit. */
int attn_fwd_fp8_ex(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                    int B, int H, int Sq, int Sk, int d, float scale,
                    float descale_q, float descale_k, float descale_v, int causal,
                    const attn_options* opts, cudaStream_t stream);

/*
 * attn_get_status — synchronises `stream`, then returns and clears the current
 * device's status word: ATTN_OK, or ATTN_ERR_TIMEOUT if any kernel launched
 * by this library on this device since the last call hit a wait limit, or
 * ATTN_ERR_LAUNCH if the synchronisation itself failed.
 */
int attn_get_status(cudaStream_t stream);

/* Static description of a status code (never NULL). */
const char* attn_strerror(int status);

/* Message of the last CUDA error seen by this thread's library calls ("" if none). */
const char* attn_last_cuda_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */

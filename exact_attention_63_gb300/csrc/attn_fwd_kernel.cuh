// Exact attention forward kernel for sm_103a (GB300).
//
// Persistent: one CTA per SM walks a list of work tiles; a tile is 128 query
// rows of one (batch, head), computed against every visible 128-key block
// with an online softmax, so the score matrix never leaves the chip
// ("FlashAttention 4: Atenção Mais Rápida …", section "Novidades no
// FlashAttention 4": blocks of Q, K, V streamed through on-chip memory).
//
// Warp roles (384 threads):
//   warp  0    loader — TMA loads of K and V tiles into a ring of shared-
//              memory slots guarded by full/empty mbarriers, in the order the
//              MMA issuers consume them (K_0 … K_{NB−1}, then V_g, K_{g+NB} for
//              every block g, across tile boundaries), so slots free up in the
//              order they are refilled; allocates and frees tensor memory
//   warp  1    P·V issuer (one thread) — tcgen05.mma O_h += P_h V_j[64h:64h+64]
//   warp  2    S issuer (one thread) — tcgen05.mma S = Q K_jᵀ
//   warp  3    Q and output (one thread) — TMA loads of each tile's Q into one
//              of two Q buffers and the TMA store of each finished tile
//   warps 4-11 softmax, two warpgroups: warpgroup h owns keys [64h, 64h+64)
//              of every 128-key block, one thread per query row (= TMEM
//              lane).  Each half is an independent online softmax with its
//              own running maximum, row sum and O accumulator; the halves are
//              merged once per tile in the epilogue with the log-sum-exp rule
//              (the merge a split over keys needs).  Splitting the columns
//              halves each thread's serial work and puts two softmax warps on
//              every scheduler, while no value crosses warpgroups per block.
//              Accumulators live in tensor memory.  An MMA issue stalls while
//              the tensor core's queue is full, so a single issuer leaves the
//              tensor core idle during each of its barrier waits; with two,
//              one issuer's waits overlap the other's MMAs.
// This is the load → MMA → softmax → rescale → store pipeline of "FlashAttention
// 4: …", section "Novidades no FlashAttention 4", with the rescale step folded
// into the softmax warps: a row is rescaled only when its block maximum
// exceeds its running maximum by more than τ (section "Reescalonamento Softmax
// Online Mais Inteligente"), which after the first blocks is rare.
//
// The schedule is built around the tensor core, which runs a 128×128×16 bf16
// MMA in 64 cycles: S has NB buffers in TMEM (two at d = 128, three at
// d = 64), so the S issuer computes S(j+1) … S(j+NB) while the softmax still
// works on S(j); the softmax seldom waits for a Q·Kᵀ, and the tensor core
// waits only for P.  Q is
// double-buffered in shared memory, so the next tile's Q arrives while the
// current tile finishes, and the issuer starts the next tile's Q·Kᵀ while the
// softmax warps write the current tile's output.
//
// The epilogue stages the tile's bf16 output in the tile's own Q buffer (idle
// once the tile's last S has completed); the store warp writes it with one TMA
// store and, once the store has read it, loads the Q of the tile two ahead
// into it.
//
// TMEM columns (512 allocated): S buffers [128·i, 128·i+128) for i < NB,
// then O_0 [128·NB, 128·NB+D) and O_1 [128·NB+D, 128·NB+2D).  P_h (bf16, two per 32-bit column) overwrites
// columns [64h, 64h+32) of its S buffer, inside the half that warpgroup h has
// already read.
//
// Ordering rules the protocol relies on:
//  * tcgen05.commit arrives only after all earlier MMAs of the committing
//    thread complete; MMAs of different threads are not ordered.  So the S
//    issuer waits for pv_done(g) — P(g)·V has completed — before S(g+NB)
//    reuses P(g)'s buffer.
//  * O_h is written by P_h(g)·V only after p_full(g), i.e. after both
//    warpgroups have finished block g (including any rescale of O_h), and a
//    rescale at block g first waits for pv_done(g−1) (the previous P·V has
//    landed).
//  * A parity wait is only correct while the barrier is within one phase of
//    the phase waited for.  Every wait here has that property: the next
//    phase needs work the waiting role has not released yet, and the
//    previous one is implied by a barrier the role already passed (when the
//    softmax sees S(g), P(g−NB)·V has completed, because S(g) was issued after
//    waiting for it).  The epilogue waits on o_final, completed once per tile
//    after its last P·V.  stage_full(b) serves the tiles staged in Q buffer
//    b; it cannot run two phases ahead of the store warp, because staging
//    tile t+2 in buffer b needs that tile's Q, which the store warp loads
//    only after its store of tile t.
//  * The K/V loader waits only for ring slots, each freed by an MMA of an
//    earlier block, so its look-ahead of NB blocks can never wait on work
//    that needs a later load.
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda.h>

#include "attn_device.cuh"

namespace attn {

constexpr int kBM = 128;       // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;       // keys per block
constexpr int kThreads = 384;  // 8 softmax warps + loader + 2 MMA issuers + output store
// The single-thread roles take the lowest warp indices: the schedulers favour
// older (lower-numbered) warps, and these warps' issue latency — above all the
// MMA issuers' — sits on the pipeline's critical path, while the softmax warps
// always have other eligible warps to overlap with.
constexpr int kLoaderWarp = 0;
constexpr int kPvWarp = 1;
constexpr int kSWarp = 2;
constexpr int kStoreWarp = 3;
constexpr int kSoftmaxWarp0 = 4;  // softmax warps 4-11
constexpr int kSoftmaxWarps = 8;
constexpr uint32_t kTmemCols = 512;
// Packed sequences without a causal mask: up to this many sequences, each
// CTA builds a prefix table of their tile counts in shared memory and walks
// only the tiles that hold rows (see tile_info).
constexpr int kSeqTableCap = 4095;
constexpr uint32_t kSeqTableBytes = (kSeqTableCap + 1) * 4;

struct FwdParams {
  void* o;                       // bf16 [B, Sq, H, D] (element strides o_sb, o_ss, o_sh)
  float* lse;                    // [B, H, Sq] ([H, total_q] for packed sequences)
  unsigned int* status;          // device status word
  unsigned long long* counters;  // optional diagnostics (may be null)
  int B, H, Sq, Sk;              // packed sequences: B = sequences, Sq = longest query sequence
  int group;                     // query heads per key/value head (H / H_kv)
  int coff;                      // causal: key j visible to row i iff j ≤ i + coff (≥ 0)
  int lse_pitch;                 // LSE elements between consecutive (batch, head) rows
  long long o_sb, o_ss, o_sh;    // element strides of O (batch, seq, head)
  // Packed sequences of different lengths (null when not): sequence s owns the
  // rows [cu_q[s], cu_q[s+1]) of Q/O and [cu_k[s], cu_k[s+1]) of K/V.
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;          // rows of the packed tensors (bounds for cu_q, cu_k)
  int bottom_right;              // packed, causal: per-sequence offset len_k − len_q
  int n_qt;                      // ceil(Sq / 128)
  int n_tiles;                   // n_qt · B · H
  float scale_log2;              // scale · log2(e)
  float tau;                     // rescale threshold, log2 domain
  float sum_limit;               // 2^tau: a half-block row sum above it sends the warp to the maximum
  float o_scale;                 // FP8 inputs: descale_v / 448 (O = o_scale · P8·V8 / L)
  uint64_t timeout_ns;
  uint32_t test_flags;           // bit 0: loader withholds K/V (exercises the wait limit)
};

template <int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kSlabs = D / 64;                 // 128-byte-wide column slabs per row
  static constexpr uint32_t kSlabBytes = kBM * 128;     // one 128-row slab: 16 KB
  static constexpr uint32_t kTileBytes = kSlabBytes * kSlabs;
  static constexpr int kStages = (D == 128) ? 4 : 10;   // K/V ring slots (each holds one K or V tile)
  // S buffers in TMEM: the S issuer runs this many blocks ahead of the
  // softmax.  Three fit at d = 64 (3·128 + 2·64 = 512 columns), two at d = 128.
  static constexpr int kSBufs = (D == 64) ? 3 : 2;
  static constexpr uint32_t kQOff = 0;                  // two Q buffers
  static constexpr uint32_t kRingOff = 2 * kTileBytes;
  // per-row (max, sum) of each half, exchanged once per tile: [tile parity][half][row] float2
  static constexpr uint32_t kStatsOff = kRingOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kStatsOff + 2 * 2 * kBM * 8;
  // barriers: q_full[2], kv_full[S], kv_empty[S], s_full[NB], p_full[NB], pv_done[NB],
  //           o_final, exch_full[2], exch_empty[2], done[2], stage_full[2]
  static constexpr int kNumBars = 2 + 2 * kStages + 3 * kSBufs + 1 + 2 + 2 + 2 + 2;
  static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;  // tmem base (4 B) + abort flag (4 B)
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base to 1024
  // (packed sequences) the sequence tile table, in the extra kSeqTableBytes
  // those launches request
  static constexpr uint32_t kTableOff = kMiscOff + 16;
  __device__ static constexpr uint32_t col_s(int buf) { return 128u * buf; }
  __device__ static constexpr uint32_t col_o(int half) {
    return 128u * kSBufs + static_cast<uint32_t>(D) * half;
  }
};


// One arrival for the whole warp: the lanes' earlier shared-memory writes (and,
// after tcgen05.wait + fence::before_thread_sync, their tensor-memory stores)
// are ordered before lane 0's release by the warp barrier.  The softmax
// barriers then take 8 arrivals a block instead of 256.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// The rescale of O_h after a row's running maximum moved at a block j > 0:
// wait until the previous P_h·V has landed in O_h, then O_h[row, :] *= alpha
// for this thread's row.  Rare after a tile's first blocks, so it is kept out
// of line: the per-block softmax code then carries neither this wait loop nor
// the scaling (inlined, they slowed the common path by several percent).
// Returns false when the wait ran out of time.
template <int D>
__device__ __noinline__ bool rescale_o(uint32_t bar_pv, uint32_t parity, WaitCtx wc, uint32_t t_o, float alpha) {
  const bool landed = wait_bar(bar_pv, parity, wc);
  if (__any_sync(0xffffffffu, !landed)) return false;
  tc_fence_after();
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(t_o + 32 * c, o);
    tmem_wait_ld();
    reg_fence32(o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
    tmem_st32(t_o + 32 * c, o);
  }
  return true;
}

// wait_bar with only the first test inline; the retry loop is a call, which
// keeps the per-block softmax code short where the barrier has usually
// completed already.
static __device__ __noinline__ bool wait_bar_retry(uint32_t bar, uint32_t parity, WaitCtx c) {
  return wait_bar(bar, parity, c);
}
__device__ __forceinline__ bool wait_bar_cold(uint32_t bar, uint32_t parity, const WaitCtx& c) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_retry(bar, parity, c);
}

// One work tile: 128 query rows of one (batch, head).
struct Tile {
  int b, h, q0, nb;  // nb = key blocks visible to the tile; < 1: the pipeline skips it
  int kvh;           // key/value head read by query head h
  int len_q, len_k;  // query rows and keys of the tile's sequence
  int coff;          // causal offset of the sequence
  int qrow, krow;    // TMA row coordinate of the tile's first query and of the sequence's first key
  int bcoord;        // TMA batch coordinate
  long long lse0;    // LSE index of the tile's first row
};

// Whether the MMA pipeline processes the tile: it has rows and sees keys
// (always, unless sequences are packed).
template <bool VARLEN>
__device__ __forceinline__ bool runs(const Tile& t) {
  if constexpr (VARLEN) return t.q0 < t.len_q && t.nb >= 1; else return true;
}

// Tile order.  Causal: heaviest query tiles first (longest-processing-time
// order for the static round-robin below).  Otherwise: the tiles of one head
// are consecutive, so CTAs working side by side share that head's K/V in L2.
//
// Packed sequences without a causal mask, given seq_tab (seq_tab[s] = H × the
// q tiles of sequences before s; seq_tab[B] = all): the index runs over the
// tiles that hold rows only, in the same order (sequence, head, q tile), so
// the round-robin over CTAs does not deal out the empty slots of sequences
// shorter than the longest (which left some CTAs with far more work).
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Tile tile_info(int idx, const FwdParams& p, const int* seq_tab = nullptr) {
  const int BH = p.B * p.H;
  int qt, bh;
  if (VARLEN && !CAUSAL && seq_tab != nullptr) {
    // The sequence s with seq_tab[s] ≤ idx < seq_tab[s+1] (it has a tile).
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seq_tab[mid] <= idx) lo = mid; else hi = mid;
    }
    const int local = idx - seq_tab[lo];
    const int c = (seq_tab[lo + 1] - seq_tab[lo]) / p.H;  // q tiles of sequence lo
    bh = lo * p.H + local / c;
    qt = local % c;
  } else if (CAUSAL) {
    qt = p.n_qt - 1 - idx / BH;
    bh = idx % BH;
  } else {
    qt = idx % p.n_qt;
    bh = idx / p.n_qt;
  }
  Tile t;
  t.b = bh / p.H;
  t.h = bh % p.H;
  t.q0 = qt * kBM;
  t.kvh = t.h / p.group;
  if constexpr (VARLEN) {
    // Packed sequences; offsets outside the tensors are clamped, so a bad
    // table cannot make the kernel read or write outside them.
    const int qa = min(max(p.cu_q[t.b], 0), p.total_q), qz = min(max(p.cu_q[t.b + 1], qa), p.total_q);
    const int ka = min(max(p.cu_k[t.b], 0), p.total_k), kz = min(max(p.cu_k[t.b + 1], ka), p.total_k);
    t.len_q = qz - qa;
    t.len_k = kz - ka;
    t.coff = (CAUSAL && p.bottom_right) ? t.len_k - t.len_q : 0;
    t.qrow = qa + t.q0;
    t.krow = ka;
    t.bcoord = 0;
    t.lse0 = static_cast<long long>(t.h) * p.lse_pitch + qa + t.q0;
    const int nk = (t.len_k + kBN - 1) / kBN;
    // Causal: the tile's last row sees keys up to row + coff (none when that
    // is negative).
    const int last = min(t.q0 + kBM, t.len_q) - 1 + t.coff;
    t.nb = CAUSAL ? (last < 0 ? 0 : min(nk, last / kBN + 1)) : nk;
  } else {
    // One sequence per batch: the sizes are the kernel's parameters (coff ≥ 0,
    // so every tile sees a key); the per-sequence fields stay unset and the
    // accessors below read the parameters instead.
    const int nk = (p.Sk + kBN - 1) / kBN;
    t.nb = CAUSAL ? min(nk, (min(t.q0 + kBM, p.Sq) - 1 + p.coff) / kBN + 1) : nk;
  }
  return t;
}

// Per-tile sizes and coordinates: from the tile for packed sequences, else
// from the kernel parameters (constant bank, no registers held).
template <bool VARLEN>
__device__ __forceinline__ int len_q_of(const Tile& t, const FwdParams& p) {
  if constexpr (VARLEN) return t.len_q; else return p.Sq;
}
template <bool VARLEN>
__device__ __forceinline__ int len_k_of(const Tile& t, const FwdParams& p) {
  if constexpr (VARLEN) return t.len_k; else return p.Sk;
}
template <bool VARLEN>
__device__ __forceinline__ int coff_of(const Tile& t, const FwdParams& p) {
  if constexpr (VARLEN) return t.coff; else return p.coff;
}
template <bool VARLEN>
__device__ __forceinline__ int qrow_of(const Tile& t) {
  if constexpr (VARLEN) return t.qrow; else return t.q0;
}
template <bool VARLEN>
__device__ __forceinline__ int krow_of(const Tile& t) {
  if constexpr (VARLEN) return t.krow; else return 0;
}
template <bool VARLEN>
__device__ __forceinline__ int bcoord_of(const Tile& t) {
  if constexpr (VARLEN) return t.bcoord; else return t.b;
}
template <bool VARLEN>
__device__ __forceinline__ long long lse0_of(const Tile& t, const FwdParams& p) {
  if constexpr (VARLEN) return t.lse0; else return (static_cast<long long>(t.b) * p.H + t.h) * p.lse_pitch + t.q0;
}

// The first tile index ≥ idx (stepping by stride) that the pipeline runs, with
// its description in T; n_tiles or more when there is none.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ int next_running(int idx, int stride, const FwdParams& p, Tile& T, int n_tiles,
                                            const int* seq_tab) {
  for (; idx < n_tiles; idx += stride) {
    T = tile_info<CAUSAL, VARLEN>(idx, p, seq_tab);
    if (runs<VARLEN>(T)) break;
  }
  return idx;
}

// Packed sequences without a causal mask (p.B <= kSeqTableCap): the prefix
// table of the sequences' q-tile counts × H, tab[s] for s in [0, B] (tab[B] =
// all tiles that hold rows), built in shared memory by every thread of the
// CTA — each sums its share of the sequences, then one scan over the lanes and
// one over the warps (warp_sums: one int per warp).  Contains __syncthreads:
// every thread of the CTA calls it.  Returns tab[B].
__device__ __forceinline__ int build_seq_table(const FwdParams& p, int* tab, int* warp_sums) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.B, nth = static_cast<int>(blockDim.x), tid = static_cast<int>(threadIdx.x);
  const int per = (n + nth - 1) / nth, s0 = min(n, tid * per), s1 = min(n, s0 + per);
  auto q_tiles = [&](int sq) {  // clamped as in tile_info; at most the n_qt tiles max_seqlen_q covers
    const int qa = min(max(p.cu_q[sq], 0), p.total_q), qz = min(max(p.cu_q[sq + 1], qa), p.total_q);
    return min((qz - qa + kBM - 1) / kBM, p.n_qt);
  };
  int mine = 0;
  for (int sq = s0; sq < s1; ++sq) mine += q_tiles(sq);
  int incl = mine;  // inclusive scan over the warp, then over the warps
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_sums[w];
  int run = before + incl - mine;
  for (int sq = s0; sq < s1; ++sq) {
    tab[sq] = run * p.H;
    run += q_tiles(sq);
  }
  if (tid == nth - 1) tab[n] = (before + incl) * p.H;
  __syncthreads();
  return tab[n];
}

// POLY: bit c selects the FMA-pipe polynomial exp2 for 16-column chunk c of
// every 128-key block (compile time, so the exp loop is one basic block).
// COUNT: compile the diagnostic counters (only launched when requested).
// VARLEN: sequences of different lengths packed along the rows.
template <int D, bool CAUSAL, uint32_t POLY, bool COUNT, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled tiles need a 1024-byte aligned base.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);

  const uint32_t sQ = base + L::kQOff;
  const uint32_t sRing = base + L::kRingOff;
  const uint32_t bars = base + L::kBarOff;
  auto bar_q_full = [&](int i) { return bars + 8u * i; };
  auto bar_kv_full = [&](int s) { return bars + 8u * (2 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (2 + L::kStages + s); };
  constexpr int NB = L::kSBufs;
  constexpr uint32_t kB0 = 2 + 2 * L::kStages;  // first per-S-buffer barrier
  auto bar_s_full = [&](int i) { return bars + 8u * (kB0 + i); };
  auto bar_p_full = [&](int i) { return bars + 8u * (kB0 + NB + i); };
  auto bar_pv_done = [&](int i) { return bars + 8u * (kB0 + 2 * NB + i); };
  const uint32_t bar_o_final = bars + 8u * (kB0 + 3 * NB);
  auto bar_exch_full = [&](int i) { return bars + 8u * (kB0 + 3 * NB + 1 + i); };
  auto bar_exch_empty = [&](int i) { return bars + 8u * (kB0 + 3 * NB + 3 + i); };
  auto bar_done = [&](int i) { return bars + 8u * (kB0 + 3 * NB + 5 + i); };
  auto bar_stage_full = [&](int i) { return bars + 8u * (kB0 + 3 * NB + 7 + i); };
  float2* const stats = reinterpret_cast<float2*>(smem + L::kStatsOff);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int stride = static_cast<int>(gridDim.x);

  // ---- set-up
  if (warp == kLoaderWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_q_full(i), 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_p_full(i), kSoftmaxWarps);  // one arrival per softmax warp
      mbar_init(bar_pv_done(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_done(i), 1);
      mbar_init(bar_exch_full(i), kSoftmaxWarps);
      mbar_init(bar_exch_empty(i), kSoftmaxWarps);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_o_final, 1);
    for (int i = 0; i < 2; ++i) mbar_init(bar_stage_full(i), kSoftmaxWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == kSWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  // Packed sequences without a causal mask: the tile prefix table (above).
  const int* seq_tab = nullptr;
  int n_tiles = p.n_tiles;
  if constexpr (VARLEN && !CAUSAL) {
    if (p.B <= kSeqTableCap) {
      int* const tab = reinterpret_cast<int*>(smem + L::kTableOff);
      n_tiles = build_seq_table(p, tab, reinterpret_cast<int*>(smem + L::kStatsOff));  // stats unused until later
      seq_tab = tab;
    }
  }

  if (warp == kLoaderWarp) {
    // =========================================================== loader
    if (lane == 0) {
      int issued = 0;  // ring loads issued
      bool ok = true;
      // Two cursors over this CTA's (tile, block) sequence, as in the issuers:
      // K runs NB blocks ahead of V.  (Q is loaded by the store warp, so this
      // thread never waits for a Q buffer: with one-block tiles, the K look-
      // ahead would otherwise wait for a store that needs a V not yet loaded.)
      Tile k_T, v_T;
      int k_idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, k_T, n_tiles, seq_tab), k_j = 0, gK = 0;
      int v_idx = k_idx, v_j = 0, gV = 0;
      v_T = k_T;
      auto ring_load = [&](const CUtensorMap* m, const Tile& T, int j) -> bool {
        const int slot = issued % L::kStages;
        if (!wait_bar(bar_kv_empty(slot), ((issued / L::kStages) & 1) ^ 1u, wc)) return false;
        mbar_arrive_expect_tx(bar_kv_full(slot), L::kTileBytes);
        for (int s = 0; s < L::kSlabs; ++s)
          tma_load_4d(sRing + slot * L::kTileBytes + s * L::kSlabBytes, m, 64 * s, T.kvh,
                      krow_of<VARLEN>(T) + j * kBN, bcoord_of<VARLEN>(T), bar_kv_full(slot));
        ++issued;
        return true;
      };
      auto load_k = [&]() -> bool {
        if (p.test_flags & 1u) return false;  // test mode: no K/V copy, the MMA wait must expire
        if (!ring_load(&tm_k, k_T, k_j)) return false;
        ++gK;
        if (++k_j == k_T.nb) {
          k_j = 0;
          k_idx = next_running<CAUSAL, VARLEN>(k_idx + stride, stride, p, k_T, n_tiles, seq_tab);
        }
        return true;
      };
      while (ok && k_idx < n_tiles && gK < gV + NB) ok = load_k();
      while (ok && v_idx < n_tiles) {
        if (!ring_load(&tm_v, v_T, v_j)) { ok = false; break; }
        ++gV;
        if (++v_j == v_T.nb) {
          v_j = 0;
          v_idx = next_running<CAUSAL, VARLEN>(v_idx + stride, stride, p, v_T, n_tiles, seq_tab);
        }
        while (ok && k_idx < n_tiles && gK < gV + NB) ok = load_k();
      }
      // Let every copy still in flight land before the CTA can exit (the
      // newest load of each slot; older ones completed before their slot was
      // refilled).
      const uint64_t t0 = globaltimer_ns();
      for (int n = (issued > L::kStages ? issued - L::kStages : 0); n < issued; ++n)
        while (!mbar_try_wait(bar_kv_full(n % L::kStages), (n / L::kStages) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else if (warp == kStoreWarp) {
    // ===================================================== output store
    // The softmax warps stage each tile's bf16 output in the tile's Q buffer;
    // one TMA store writes it (rows beyond Sq are clipped).  The same thread
    // loads the Q tiles: the CTA's first two at the start, then tile t+2's
    // into tile t's buffer as soon as the store of tile t has read it.
    // Doing this here keeps the store's latency off the softmax warps and the
    // Q buffers' turnover off the K/V loader.
    if (lane == 0) {
      Tile Tq;
      int q_idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, Tq, n_tiles, seq_tab), q_issued = 0;
      auto load_q = [&]() {
        const int qb = q_issued & 1;
        mbar_arrive_expect_tx(bar_q_full(qb), L::kTileBytes);
        for (int sl = 0; sl < L::kSlabs; ++sl)
          tma_load_4d(sQ + qb * L::kTileBytes + sl * L::kSlabBytes, &tm_q, 64 * sl, Tq.h, qrow_of<VARLEN>(Tq),
                      bcoord_of<VARLEN>(Tq), bar_q_full(qb));
        ++q_issued;
        q_idx = next_running<CAUSAL, VARLEN>(q_idx + stride, stride, p, Tq, n_tiles, seq_tab);
      };
      for (int n = 0; n < 2 && q_idx < n_tiles; ++n) load_q();
      int tc = 0;
      Tile T;
      for (int idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, T, n_tiles, seq_tab); idx < n_tiles;
           idx = next_running<CAUSAL, VARLEN>(idx + stride, stride, p, T, n_tiles, seq_tab), ++tc) {
        const int qb = tc & 1;
        if (!wait_bar(bar_stage_full(qb), (tc >> 1) & 1, wc)) break;
        // A packed sequence's last tile is written by the softmax threads
        // (its rows beyond the sequence belong to the next one).
        if (!VARLEN || T.q0 + kBM <= len_q_of<VARLEN>(T, p)) {
          for (int sl = 0; sl < L::kSlabs; ++sl)
            tma_store_4d(&tm_o, sQ + qb * L::kTileBytes + sl * L::kSlabBytes, 64 * sl, T.h, qrow_of<VARLEN>(T),
                         bcoord_of<VARLEN>(T));
          tma_store_commit();
          tma_store_wait_read0();
        }
        if (q_idx < n_tiles) load_q();  // tile tc + 2, into buffer qb
      }
      // Let the Q copies still in flight land before the CTA can exit.
      const uint64_t t0 = globaltimer_ns();
      for (int n = (q_issued > 2 ? q_issued - 2 : 0); n < q_issued; ++n)
        while (!mbar_try_wait(bar_q_full(n & 1), (n >> 1) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else if (warp == kSWarp || warp == kPvWarp) {
    // ====================================================== MMA issuers
    // Ring positions follow the loader's order K_0 … K_{NB−1}, then V_g,
    // K_{g+NB} per block g, then the remaining V's, over the CTA's G blocks:
    // K_j → j for j < NB, else 2j − NB + 1; V_g → min(2g + NB, G + g).
    if (lane == 0) {
      bool ok = true;
      if (warp == kSWarp) {
        // ------------------------------------------------------ S issuer
        constexpr uint32_t idS = idesc_bf16(kBM, kBN, false);
        // Descriptor bases, computed once; each operand is a base plus a
        // constant (start address in 16-byte units; shared-memory offsets
        // stay below 256 KB, so the 14-bit field never carries).
        const uint64_t dQ = sdesc_kmajor_sw128(sQ);
        const uint64_t dK = sdesc_kmajor_sw128(sRing);
        int g = 0, tc = 0;
        Tile T;
        for (int idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, T, n_tiles, seq_tab); idx < n_tiles && ok;
             idx = next_running<CAUSAL, VARLEN>(idx + stride, stride, p, T, n_tiles, seq_tab), ++tc) {
          const int qb = tc & 1;
          for (int j = 0; j < T.nb; ++j, ++g) {
            const int buf = g % NB;
            // Operands first: Q and K_j arrive well ahead, so these waits stay
            // off the softmax → P·V → S chain.  (K_j's ring slot was freed by
            // an S this thread has already issued, so waiting here first
            // cannot block that chain.)
            if (j == 0 && !wait_bar(bar_q_full(qb), (tc >> 1) & 1, wc)) { ok = false; break; }
            const int n = (g < NB) ? g : 2 * g - NB + 1, slot = n % L::kStages;
            if (!wait_bar(bar_kv_full(slot), (n / L::kStages) & 1, wc)) { ok = false; break; }
            // S(g) reuses the buffer of P(g−NB): that P·V must have completed.
            if (g >= NB && !wait_bar(bar_pv_done(buf), ((g - NB) / NB) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dq = dQ + ((qb * L::kTileBytes) >> 4);
            const uint64_t dk = dK + ((slot * L::kTileBytes) >> 4);
            const uint32_t tS = tmem + L::col_s(buf);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk / 4) * L::kSlabBytes + (kk % 4) * 32) >> 4;
              mma_ss(tS, dq + off, dk + off, idS, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar_s_full(buf));
            mma_commit(bar_kv_empty(slot));                     // K_j no longer read
            // (The tile's Q buffer is released by the epilogue, which reuses it.)
          }
        }
      } else {
        // ---------------------------------------------------- P·V issuer
        constexpr uint32_t idPV = idesc_bf16(kBM, D, true);
        const uint64_t dV = sdesc_mnmajor_sw128(sRing, L::kSlabBytes);
        Tile T;
        int G = 0;  // blocks of this CTA
        for (int idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, T, n_tiles, seq_tab); idx < n_tiles;
             idx = next_running<CAUSAL, VARLEN>(idx + stride, stride, p, T, n_tiles, seq_tab))
          G += T.nb;
        int g = 0;
        for (int idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, T, n_tiles, seq_tab); idx < n_tiles && ok;
             idx = next_running<CAUSAL, VARLEN>(idx + stride, stride, p, T, n_tiles, seq_tab)) {
          for (int j = 0; j < T.nb; ++j, ++g) {
            const int buf = g % NB;
            // V_j first (loaded well ahead; its slot was freed by a P·V this
            // thread already issued), then the softmax's P(g).
            const int n = min(2 * g + NB, G + g), slot = n % L::kStages;
            if (!wait_bar(bar_kv_full(slot), (n / L::kStages) & 1, wc)) { ok = false; break; }
            if (!wait_bar(bar_p_full(buf), (g / NB) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            // O_h (+)= P_h(g) · V_j[64h : 64h+64]
            const uint64_t dv = dV + ((slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t tP = tmem + L::col_s(buf) + 64 * h;
              const uint32_t tOh = tmem + L::col_o(h);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(tOh, tP + kk * 8, dv + (((4 * h + kk) * 2048) >> 4), idPV, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar_pv_done(buf));
            if (j == T.nb - 1) mma_commit(bar_o_final);  // the tile's O_0, O_1 are complete
            mma_commit(bar_kv_empty(slot));                // V_j no longer read
          }
        }
      }
      // Every MMA this thread issued must finish before TMEM is released.
      const int me = warp - kPvWarp;
      mma_commit(bar_done(me));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_done(me), 0))
        if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else {
    // ========================================================== softmax
    const int h = (warp - kSoftmaxWarp0) >> 2;  // key half owned by this warpgroup
    const int r = threadIdx.x & 127;  // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tOh = tmem + L::col_o(h) + lane_off;
    const float sc = p.scale_log2;
    const uint64_t sc2 = pack2(sc, sc);
    constexpr int kHalf = kBN / 2;  // keys per half
    bool ok = true;
    int g = 0;   // global block counter of this CTA
    int tc = 0;  // tiles of this CTA the pipeline has run
    // O row of this thread in tile T (element offset), for the tiles the
    // softmax threads write directly.
    auto o_row = [&](const Tile& T) -> uint16_t* {
      return static_cast<uint16_t*>(p.o) + bcoord_of<VARLEN>(T) * p.o_sb +
             static_cast<long long>(qrow_of<VARLEN>(T) + r) * p.o_ss + T.h * p.o_sh;
    };
    for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride) {
      const Tile T = tile_info<CAUSAL, VARLEN>(idx, p, seq_tab);
      const int q_row = T.q0 + r;
      if constexpr (VARLEN) {
        if (!runs<VARLEN>(T)) {
          // A tile beyond its sequence has nothing to write; rows of a tile
          // that sees no key get O = 0 and LSE = −inf.
          if (T.q0 < T.len_q && q_row < T.len_q) {
            uint4* const dst = reinterpret_cast<uint4*>(o_row(T) + h * (D / 2));
#pragma unroll
            for (int c = 0; c < D / 16; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            if (h == 0) p.lse[T.lse0 + r] = -INFINITY;
          }
          continue;
        }
      }
      float m_run = -INFINITY;  // running reference maximum of this half (log2 domain)
      float l_run = 0.f;        // running row sum of this half (fp32, unrounded p)
      // Row maximum of this half (log2 domain): four independent 16-wide chains.
      auto row_max = [&](const float* x0) -> float {
        float m4[4];
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const float* x = x0 + 16 * gg;
          float a = fmax3(x[0], x[1], x[2]);
          float b2 = fmax3(x[3], x[4], x[5]);
          a = fmax3(a, x[6], x[7]);
          b2 = fmax3(b2, x[8], x[9]);
          a = fmax3(a, x[10], x[11]);
          b2 = fmax3(b2, x[12], x[13]);
          m4[gg] = fmax3(a, b2, fmaxf(x[14], x[15]));
        }
        return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sc;
      };
      // p = 2^(s·scale·log2 e − m_run) for this half's 64 keys: bf16 pairs in
      // pk, the fp32 sum of the unrounded values returned.
      auto exps = [&](const float* s, uint32_t (&pk)[kHalf / 2]) -> float {
        const float negm = (m_run == -INFINITY) ? 0.f : -m_run;
        const uint64_t nm2 = pack2(negm, negm);
        uint64_t acc[4] = {0, 0, 0, 0};  // four packed partial sums (+0.0f pairs)
#pragma unroll
        for (int ch = 0; ch < kHalf / 16; ++ch) {
          constexpr uint32_t kPoly = POLY;
          const bool use_poly = (kPoly >> (4 * h + ch)) & 1u;  // folded after unrolling
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = ch * 16 + 2 * i;
            float x0, x1;
            unpack2(ffma2(pack2(s[c], s[c + 1]), sc2, nm2), x0, x1);
            if (use_poly) {
              ex2_poly2(x0, x1);
            } else {
              x0 = ex2_mufu(x0);
              x1 = ex2_mufu(x1);
            }
            acc[i & 3] = fadd2(acc[i & 3], pack2(x0, x1));
            pk[ch * 8 + i] = pack_bf16x2(x0, x1);
          }
        }
        float a0, a1, b0, b1;
        unpack2(fadd2(acc[0], acc[1]), a0, a1);
        unpack2(fadd2(acc[2], acc[3]), b0, b1);
        return (a0 + a1) + (b0 + b1);
      };
      // One key block.  MASK selects the copy that masks keys beyond Sk and,
      // when causal, keys after the row; only the tile's last blocks need it,
      // so the loop over the other blocks runs a copy without that code.
      auto block = [&](int j, auto mask_tag) -> bool {
        constexpr bool MASK = decltype(mask_tag)::value;
        const int buf = g % NB;
        const uint32_t tS = tmem + L::col_s(buf) + kHalf * h + lane_off;
        const bool got = wait_bar_cold(bar_s_full(buf), (g / NB) & 1, wc);
        if (__any_sync(0xffffffffu, !got)) return false;
        tc_fence_after();
        // This half of the S row (64 fp32) in registers: two loads, one wait.
        uint32_t u[kHalf];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tmem_wait_ld();
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        float* const s = reinterpret_cast<float*>(u);
        if constexpr (MASK) {
          const int k0 = j * kBN + kHalf * h;
#pragma unroll
          for (int c = 0; c < kHalf; ++c) {
            const int key = k0 + c;
            if (key >= len_k_of<VARLEN>(T, p) || (CAUSAL && key > q_row + coff_of<VARLEN>(T, p))) s[c] = -INFINITY;
          }
        }
        // The exponentials are taken straight away against the running
        // reference maximum.  Only when a row has no reference yet (its first
        // visible block), or when its half-block sum shows a key far above the
        // reference (Σp > 2^τ, so some p may exceed 2^τ; this also catches an
        // overflow to inf), does the warp compute the block maximum, rescale
        // where the maximum moved by more than τ, and redo the exponentials.
        // The outputs are those of computing the maximum first: a row that
        // passes the sum test has no key above m_run + τ, so it would not
        // have been rescaled.  After a tile's first block the sum test almost
        // never fails, so the maximum leaves the per-block path.
        uint32_t pk[kHalf / 2];
        float lsum;
        bool redo = __any_sync(0xffffffffu, m_run == -INFINITY);
#pragma unroll 1
        for (;;) {
          if (redo) {
            const float mx = row_max(s);
            const bool need = mx > m_run + p.tau;
            if (__any_sync(0xffffffffu, need)) {
              const float m_new = need ? mx : m_run;
              const float alpha = need ? ex2_mufu(m_run - m_new) : 1.f;
              // O_h holds the tile's blocks < j once the last P_h·V has landed.
              if (j > 0 && !rescale_o<D>(bar_pv_done((g - 1) % NB), ((g - 1) / NB) & 1, wc, tOh, alpha))
                return false;
              l_run *= alpha;
              m_run = m_new;
              if constexpr (COUNT) {
                const unsigned int nres = __popc(__ballot_sync(0xffffffffu, need));
                if (lane == 0) atomicAdd(p.counters, static_cast<unsigned long long>(nres));
              }
            }
            __syncwarp();
          }
          lsum = exps(s, pk);
          if (redo || !__any_sync(0xffffffffu, !(lsum <= p.sum_limit))) break;
          redo = true;
        }
        if constexpr (COUNT) {
          if (lane == 0 && h == 0) atomicAdd(p.counters + 1, 32ull);
        }
        tmem_st32(tS, pk);  // P_h over the first 32 columns of this half
        l_run += lsum;
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar_p_full(buf), lane);
        return true;
      };
      // Block j needs no mask for this half when all its keys lie below lim
      // (Sk, and when causal also the tile's first row + coff + 1):
      // 128j + 64h + 64 ≤ lim, i.e. j < (lim − 64h + 64) / 128.
      const int lk = len_k_of<VARLEN>(T, p);
      const int lim = CAUSAL ? min(lk, T.q0 + 1 + coff_of<VARLEN>(T, p)) : lk;
      const int n_full = min(T.nb, max(0, (lim - kHalf * h + kHalf) / kBN));
      int j = 0;
      for (; j < n_full && ok; ++j, ++g) ok = block(j, std::false_type{});
      for (; j < T.nb && ok; ++j, ++g) ok = block(j, std::true_type{});
      if (!ok) break;
      // ---------------------------------------------------- epilogue
      // Exchange (max, sum) with the other half's thread of the same row.
      const int par = tc & 1;
      {
        const bool free_ = wait_bar(bar_exch_empty(par), ((tc >> 1) & 1) ^ 1u, wc);
        if (__any_sync(0xffffffffu, !free_)) { ok = false; break; }
      }
      stats[(par * 2 + h) * kBM + r] = make_float2(m_run, l_run);
      warp_arrive(bar_exch_full(par), lane);
      {
        const bool in = wait_bar(bar_exch_full(par), (tc >> 1) & 1, wc);
        if (__any_sync(0xffffffffu, !in)) { ok = false; break; }
      }
      const float2 other = stats[(par * 2 + (h ^ 1)) * kBM + r];
      warp_arrive(bar_exch_empty(par), lane);
      // Merge the halves: m = max, a_i = 2^(m_i − m), L = Σ a_i l_i.
      const float m0 = h ? other.x : m_run, l0 = h ? other.y : l_run;
      const float m1 = h ? m_run : other.x, l1 = h ? l_run : other.y;
      const float m = fmaxf(m0, m1);
      const float a0 = (m0 == -INFINITY) ? 0.f : ex2_mufu(m0 - m);
      const float a1 = (m1 == -INFINITY) ? 0.f : ex2_mufu(m1 - m);
      const float Lsum = a0 * l0 + a1 * l1;
      const float inv = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
      const float w0 = a0 * inv, w1 = a1 * inv;
      // The tile's last P·V completes phase tc of o_final.
      const bool landed = wait_bar(bar_o_final, tc & 1, wc);
      if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }
      tc_fence_after();
      // Warpgroup h produces output columns [h·D/2, (h+1)·D/2), staged in the
      // tile's Q buffer with the 128-byte swizzle the TMA store expects (16-byte
      // chunk c of row r at c ^ (r % 8): conflict-free for 8 consecutive rows).
      const uint32_t t0 = tmem + L::col_o(0) + lane_off + h * (D / 2);
      const uint32_t t1 = tmem + L::col_o(1) + lane_off + h * (D / 2);
      const int qb = tc & 1;
      uint8_t* const stage = smem + L::kQOff + qb * L::kTileBytes;
      // A packed sequence's last tile: each thread writes its own row (rows
      // beyond the sequence belong to the next one); else staged for the TMA
      // store.
      const bool direct = VARLEN && T.q0 + kBM > len_q_of<VARLEN>(T, p);
      uint16_t* const orow = o_row(T);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t x0[32], x1[32];
        tmem_ld32(t0 + 32 * c, x0);
        tmem_ld32(t1 + 32 * c, x1);
        tmem_wait_ld();
        reg_fence32(x0);
        reg_fence32(x1);
#pragma unroll
        for (int q16 = 0; q16 < 4; ++q16) {  // four 16-byte chunks of 8 values
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            v[e] = w0 * __uint_as_float(x0[8 * q16 + e]) + w1 * __uint_as_float(x1[8 * q16 + e]);
          uint4 wv;
          wv.x = pack_bf16x2(v[0], v[1]);
          wv.y = pack_bf16x2(v[2], v[3]);
          wv.z = pack_bf16x2(v[4], v[5]);
          wv.w = pack_bf16x2(v[6], v[7]);
          const int col = h * (D / 2) + 32 * c + 8 * q16;
          const int chunk = (col & 63) >> 3;
          if (!direct)
            *reinterpret_cast<uint4*>(stage + (col >> 6) * L::kSlabBytes + r * 128 + ((chunk ^ (r & 7)) << 4)) = wv;
          else if (q_row < len_q_of<VARLEN>(T, p))
            *reinterpret_cast<uint4*>(orow + col) = wv;
        }
      }
      fence_proxy_async_smem();
      warp_arrive(bar_stage_full(qb), lane);  // the store warp writes the tile out
      if (h == 0 && q_row < len_q_of<VARLEN>(T, p)) {
        const float lse = (Lsum > 0.f) ? (m + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        p.lse[lse0_of<VARLEN>(T, p) + r] = lse;
      }
      ++tc;
    }
  }

  // ---- tear-down: every role arrives here; all TMEM reads/writes are done
  tc_fence_before();
  __syncthreads();
  if (warp == kLoaderWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn

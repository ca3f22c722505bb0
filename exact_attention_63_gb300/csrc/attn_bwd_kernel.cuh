// Exact attention backward kernels for sm_103a (GB300).
//
// Gradients of O = softmax(scale·QKᵀ)V for a loss with dL/dO = dO, from the
// forward's O and LSE: with P = exp(scale·QKᵀ − LSE) over visible keys,
//   dV = Pᵀ dO,  dP = dO Vᵀ,  D = rowsum(dO ∘ O),  dS = P ∘ (dP − D),
//   dQ = scale · dS K,  dK = scale · dSᵀ Q.
// (The pages give no backward formulas; "FlashAttention-4 no Blackwell B200
// …", section "Redução de tráfego no backward", says FA4 keeps the backward's
// intermediates in tensor memory.  These kernels do that too: S, dP, P, dS and
// the accumulators live in TMEM, and P / dS feed the MMAs from there.)
//
// One kernel template serves the two passes and the fused one; a CTA owns one tile of 128 rows of
// one (batch, head) and walks the blocks of 128 columns that the rows see:
//   DQ  rows = queries (X = Q, X2 = dO), columns = keys  (A = K, B = V):
//       S = Q Kᵀ, dP = dO Vᵀ, P and dS per (query, key), dQ += dS K.
//   DKV rows = keys (X = K, X2 = V), columns = queries (A = Q, B = dO):
//       Sᵀ = K Qᵀ, dPᵀ = V dOᵀ, Pᵀ and dSᵀ per (key, query),
//       dV += Pᵀ dO, dK += dSᵀ Q.
// With grouped key/value heads the dQ pass reads the K/V head of its query
// head's group, and the dK/dV (and fused) pass of a K/V head walks the query blocks of
// every query head in its group (their contributions add up).
//   FUSED (d = 64) rows = keys, as DKV, and dQ in the same pass: dS goes to a
//       shared-memory tile (not over dP), dK += dSᵀ Q reads it K-major and
//       dQ(n) = dS K — the block's contribution to its 128 queries' dQ —
//       reads it MN-major; the warps add dQ(n) into an fp32 accumulator in
//       device memory by TMA reduce-add, and a last kernel rounds it to bf16.
//       S and dP are then computed once per (query, key) pair instead of
//       twice, at the price of an accumulation order that varies from run to
//       run (fp32 additions of the key tiles' contributions).
// In all, S = X·Aᵀ and dP = X2·Bᵀ are K-major products like the forward's
// Q·Kᵀ, and every accumulation is TMEM operand × MN-major shared-memory
// operand like the forward's P·V, except the fused pass's dK and dQ, whose
// dS operand is in shared memory.  DQ and DKV use no atomics (separate
// passes; bit-reproducible).
//
// Warp roles (352 threads): warps 0-7 turn S, dP into P, dS (warpgroup h owns
// columns [64h, 64h+64) of each block; one thread per row) and write the
// tile's outputs; warp 8 loads X, X2 once and streams (A, B) blocks — plus, in
// DKV, the 128 −log2-LSE and D values of the block's queries — through a ring;
// warp 9 issues S and dP, warp 10 the accumulations.  One thread issues at
// most one tcgen05.mma every ~45 cycles (more beside busy warps): a block is
// 24 (d = 64) to 32 (d = 128) MMAs, about as long as the tensor core's own
// work on them, so the issue is split; every dependency between the two
// threads' MMAs goes through a completion barrier, and each accumulator is
// written by one thread only (in issue order).
//
// Schedule.  A shared-memory-operand MMA reads both of its tiles at the
// shared-memory rate (128 B/clk per SM: a 128×128×16 product takes its 64
// cycles, a 128×64×16 one 48 instead of 32), so S and dP are each computed
// for all 128 columns at once and the rest of the block is pipelined around
// them with TMEM-operand accumulations (which read only their B tile):
//   DKV: S(n), dP(n); the warpgroups store P over S and signal per half, so
//        dV += Pᵀ dO starts while they form dS; dK += dSᵀ Q per half as dS
//        lands over dP.  S(n+1) waits for dV(n) (it overwrites P(n)), dP(n+1)
//        for dK(n).
//   DQ:  S(n), dP(n); the warpgroups read S and release its columns at once
//        (P stays in registers), so S(n+1) overlaps their work; dS goes to
//        columns of its own (free in this pass) and dQ += dS K runs per half;
//        dP(n+1) follows as soon as the warps have read dP(n).
//
// TMEM columns: S [0, 128), dP [128, 256), acc0 [256, 256+D) (dQ or dV),
// acc1 [256+D, 256+2D) (dK; in the dQ pass two 64-column dS buffers), and in
// the dK/dV and fused passes at d = 64 a second S buffer [384, 512) (S(n+1)
// then waits for dV(n−1), not dV(n)).  P (bf16 pairs)
// overwrites S's columns and, in DKV, dS overwrites dP's, in the packed layout
// the forward uses for P.  The fused pass's dQ(n) goes to S(n)'s columns
// [32, 96) (P's two halves are packed into [0, 32) and [96, 128) there).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "attn_bwd_launch.h"
#include "attn_device.cuh"

namespace attn {

constexpr int kBwdThreads = 352;
constexpr int kBwdLoaderWarp = 8;
constexpr int kBwdMmaWarp = 9;   // S and dP
constexpr int kBwdAccWarp = 10;  // the accumulations (dV, dK or dQ)
constexpr int kModeDQ = 0;
constexpr int kModeDKV = 1;
constexpr int kModeFused = 2;


template <int D, int MODE>
struct BwdLayout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr bool kKeys = (MODE != kModeDQ);  // rows are keys (dK/dV and fused passes)
  static constexpr bool kFused = (MODE == kModeFused);
  static constexpr int kSlabs = D / 64;
  static constexpr uint32_t kSlabBytes = 128 * 128;
  static constexpr uint32_t kTileBytes = kSlabBytes * kSlabs;
  static constexpr int kStages = (D == 128) ? 2 : 3;
  static constexpr uint32_t kVecBytes = kKeys ? 2 * 128 * 4 : 0;  // −log2-LSE and D of 128 queries
  static constexpr uint32_t kSlotBytes = 2 * kTileBytes + ((kVecBytes + 1023) / 1024) * 1024;
  static constexpr uint32_t kXOff = 0;                       // X, X2
  static constexpr uint32_t kRingOff = 2 * kTileBytes;
  // The fused pass is built for d = 64: at d = 128 S, dP and the two
  // accumulators take all of TMEM, so dQ(n) would have to share dP's columns
  // (dP(n+1) then waits for dQ(n)'s read-out), no staging buffer fits beside
  // the dS tile, and its reduce-adds bound it (slower than the two passes).
  static_assert(!kFused || D == 64, "the fused pass is built for d = 64");
  // Fused pass: the dS tile, 128 keys × 128 queries bf16 in two 64-query
  // slabs with the 128-byte swizzle (K-major for dK, MN-major for dQ), and
  // the fp32 dQ(n) staging (128 × 64: two spans of 128 rows × 32 values,
  // 128-byte swizzle), a buffer of its own: the warps never wait for the
  // reduce-adds to read it before going on, only before they restage their
  // rows a block later.
  static constexpr uint32_t kDSOff = kRingOff + kStages * kSlotBytes;
  static constexpr uint32_t kStageOff = kDSOff + (kFused ? 2 * kSlabBytes : 0);
  static constexpr uint32_t kStageBytes = (D / 32) * 128 * 128;
  static constexpr uint32_t kTilesBytes = kStageOff + (kFused ? kStageBytes : 0);
  // barriers: fix_full, ring_full[S], ring_empty[S], s_full, dp_full, p_full[2], ds_full[2][2],
  //           acc_a, acc_b, done, dq_done[2], s_full_1, acc_a_1, p_full_1[2], dq_full, dq_free, dp_read
  static constexpr int kNumBars = 1 + 2 * kStages + 20;
  // The dK/dV and fused passes at d = 64 leave TMEM columns [384, 512) free:
  // S gets a second buffer there, so S(n+1) does not wait for dV(n).
  static constexpr bool kDblS = (kKeys && D == 64);
  // The barriers and words (under 512 B) sit below the 1024-byte-aligned
  // tiles when the alignment gap holds them, else right after the tiles:
  // both fit in tiles + 1024 bytes.
  static constexpr uint32_t kMiscOff = 8 * kNumBars;  // within the barrier block
  static constexpr uint32_t kMetaBytes = kMiscOff + 16;
  static_assert(kMetaBytes <= 512, "the barrier block fits below the tiles or after them");
  static constexpr uint32_t kSmemBytes = kTilesBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

template <int D, bool CAUSAL, int MODE>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_x2,
                    const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_o0, const __grid_constant__ CUtensorMap tm_o1,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using L = BwdLayout<D, MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);
  // base − raw < 1024: the barrier block goes below base when it fits there,
  // else after the tiles (then base − raw < kMetaBytes ≤ 1024 − kMetaBytes).
  const uint32_t meta = (base - raw >= L::kMetaBytes) ? raw : base + L::kTilesBytes;
  uint8_t* const meta_ptr = smem_raw + (meta - raw);
  const uint32_t sX = base + L::kXOff;
  const uint32_t sRing = base + L::kRingOff;
  const uint32_t sDS = base + L::kDSOff;
  const uint32_t bars = meta;
  const uint32_t bar_fix = bars;
  auto bar_ring_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_ring_empty = [&](int s) { return bars + 8u * (1 + L::kStages + s); };
  const uint32_t bar_b0 = bars + 8u * (1 + 2 * L::kStages);
  // S of block n written, and (DKV) dV(n) done (its S buffer is free): with
  // two S buffers, one barrier of each per buffer (phase n >> 1), so that
  // neither runs two phases ahead of its waiter; else one (phase n).
  auto bar_s_full = [&](int n) { return (L::kDblS && (n & 1)) ? bar_b0 + 8u * 13 : bar_b0; };
  auto s_par = [](int n) { return static_cast<uint32_t>(L::kDblS ? (n >> 1) : n) & 1u; };
  const uint32_t bar_dp_full = bar_b0 + 8u;      // dP of the block written
  // DKV: P of a half stored over S; DQ: S of a half read (its columns are free)
  // (with two S buffers: one barrier per half and block parity, phase n >> 1;
  // P(n+2) needs S(n+2), which waits for dV(n), the first waiter's work)
  auto bar_p_full = [&](int hh, int n) {
    return (L::kDblS && (n & 1)) ? bar_b0 + 8u * (15 + hh) : bar_b0 + 8u * (2 + hh);
  };
  // dS of a half stored (so dP of the half has been read)
  // dS of half hh of block n stored (so dP of the half has been read):
  // barrier (hh, n & 1), phase n >> 1.  Two waiters (the S/dP issuer in DQ,
  // the accumulation issuer in both passes) and one barrier per block parity:
  // dS(n+2) is stored only after dQ(n) (DQ: the dS buffer) or dK(n+1) (DKV:
  // dP(n+2) waits for it), so neither waiter can fall two phases behind.
  auto bar_ds_full = [&](int hh, int n) { return bar_b0 + 8u * (4 + 2 * hh + (n & 1)); };
  auto ds_par = [](int n) { return static_cast<uint32_t>(n >> 1) & 1u; };
  auto bar_acc_a = [&](int n) { return (L::kDblS && (n & 1)) ? bar_b0 + 8u * 14 : bar_b0 + 8u * 8; };
  const uint32_t bar_acc_b = bar_b0 + 8u * 9;    // DKV: dK of the block done (dP's columns are free)
  const uint32_t bar_done = bar_b0 + 8u * 10;    // every MMA done
  // DQ: dQ of the blocks using dS buffer i done (that buffer is free); one
  // barrier per buffer, so each is waited on one phase at a time
  auto bar_dq_done = [&](int i) { return bar_b0 + 8u * (11 + i); };
  // Fused: dV(n), dK(n) and dQ(n) done (one commit after dQ(n): block n's
  // slot and the dS tile are no longer read, dQ(n) can be read out); and
  // dQ(n) read out of TMEM by all eight warps (its columns are free).  One
  // barrier each, phase n: the warps read dQ(n) before they store dS(n+1),
  // which dQ(n+1) waits for, and S(n+2) — in dQ(n)'s S buffer — waits for
  // dQ(n)'s release before the warps can reach dQ(n+1).
  const uint32_t bar_dq_full = bar_b0 + 8u * 17;
  const uint32_t bar_dq_free = bar_b0 + 8u * 18;
  // Fused and dQ passes: dP(n) read by all eight warps (its columns may take
  // dP(n+1); dS has a place of its own); phase n: dP(n+1), which the next
  // phase needs, waits for it.
  const uint32_t bar_dp_read = bar_b0 + 8u * 19;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(meta_ptr + L::kMiscOff);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(meta_ptr + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- the tile and the blocks of 128 columns its rows see
  const int h_rows = (MODE == kModeDQ) ? p.H : p.H / p.group;  // heads of the row tensor
  const int rt = blockIdx.x % p.n_rt;
  const int bh = blockIdx.x / p.n_rt;
  const int b = bh / h_rows, h = bh % h_rows;  // h: query head (dQ) or key/value head (dK/dV)
  const int r0 = rt * 128;
  const int n_q = (p.Sq + 127) / 128, n_k = (p.Sk + 127) / 128;
  int c_first, c_end;  // column blocks [c_first, c_end)
  if (MODE == kModeDQ) {
    c_first = 0;
    c_end = CAUSAL ? min(n_k, (min(r0 + 128, p.Sq) - 1 + p.coff) / 128 + 1) : n_k;
  } else {
    // Queries i see key j iff j ≤ i + coff: the tile's first key r0 is first
    // seen by query r0 − coff.
    c_first = CAUSAL ? max(0, (r0 - p.coff) / 128) : 0;
    if (CAUSAL && r0 - p.coff < 0) c_first = 0;
    c_end = n_q;
  }
  if (c_end < c_first) c_end = c_first;
  // The dK/dV pass walks its column blocks once per query head of the group.
  const int n_per = c_end - c_first;
  const int nblk = L::kKeys ? n_per * p.group : n_per;
  // Column block n: its first column, and the head of the A/B tensors.
  auto col0_of = [&](int n) { return (c_first + (L::kKeys ? n % max(n_per, 1) : n)) * 128; };
  auto head_of = [&](int n) { return L::kKeys ? h * p.group + n / max(n_per, 1) : h / p.group; };

  if (warp == kBwdLoaderWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar_fix, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_ring_full(s), 1);
      mbar_init(bar_ring_empty(s), 1);  // the accumulation issuer's commit
    }
    mbar_init(bar_s_full(0), 1);
    mbar_init(bar_s_full(1), 1);
    mbar_init(bar_dp_full, 1);
    for (int hh = 0; hh < 2; ++hh) {
      mbar_init(bar_p_full(hh, 0), 4);  // one arrival per warp of the half's warpgroup
      mbar_init(bar_p_full(hh, 1), 4);
      mbar_init(bar_ds_full(hh, 0), 4);
      mbar_init(bar_ds_full(hh, 1), 4);
    }
    mbar_init(bar_acc_a(0), 1);
    mbar_init(bar_acc_a(1), 1);
    mbar_init(bar_acc_b, 1);
    mbar_init(bar_done, 2);  // one commit per issuing thread
    for (int i = 0; i < 2; ++i) mbar_init(bar_dq_done(i), 1);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_free, 8);  // one arrival per gradient warp
    mbar_init(bar_dp_read, 8);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const uint32_t tdP = tmem + 128, tAcc0 = tmem + 256, tAcc1 = tmem + 256 + D;
  auto tS = [&](int n) { return tmem + ((L::kDblS && (n & 1)) ? 384u : 0u); };  // S (and P) of block n
  // dQ pass: dS gets columns of its own (where dK sits in the other pass), two
  // buffers of 64, so neither the next block's dP nor its dS waits for the
  // previous dQ += dS K.
  auto tDS = [&](int n) { return tAcc1 + 64u * (n & 1); };
  // Fused pass: dQ(n) in S(n)'s free middle columns; P's half hh packed at
  // column pcol(hh) of S's buffer.
  auto tQ = [&](int n) { return tS(n) + 32u; };
  auto pcol = [](int hh) { return static_cast<uint32_t>(64 * hh + ((L::kFused && hh) ? 32 : 0)); };

  if (warp == kBwdLoaderWarp) {
    // ============================================================ loader
    if (lane == 0 && nblk > 0) {
      mbar_arrive_expect_tx(bar_fix, 2 * L::kTileBytes);
      for (int s = 0; s < L::kSlabs; ++s) {
        tma_load_4d(sX + s * L::kSlabBytes, &tm_x, 64 * s, h, r0, b, bar_fix);
        tma_load_4d(sX + L::kTileBytes + s * L::kSlabBytes, &tm_x2, 64 * s, h, r0, b, bar_fix);
      }
      int n = 0;
      for (; n < nblk; ++n) {
        const int slot = n % L::kStages;
        if (!wait_bar(bar_ring_empty(slot), ((n / L::kStages) & 1) ^ 1u, wc)) break;
        const uint32_t dst = sRing + slot * L::kSlotBytes;
        const int c0 = col0_of(n), ha = head_of(n);
        mbar_arrive_expect_tx(bar_ring_full(slot), 2 * L::kTileBytes + L::kVecBytes);
        for (int s = 0; s < L::kSlabs; ++s) {
          tma_load_4d(dst + s * L::kSlabBytes, &tm_a, 64 * s, ha, c0, b, bar_ring_full(slot));
          tma_load_4d(dst + L::kTileBytes + s * L::kSlabBytes, &tm_b, 64 * s, ha, c0, b, bar_ring_full(slot));
        }
        if (L::kKeys) {
          const size_t row = (static_cast<size_t>(b) * p.H + ha) * p.pitch + c0;
          bulk_load(dst + 2 * L::kTileBytes, p.lse2 + row, 512, bar_ring_full(slot));
          bulk_load(dst + 2 * L::kTileBytes + 512, p.dvec + row, 512, bar_ring_full(slot));
        }
      }
      // Let the copies in flight land before the CTA can exit.
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_fix, 0))
        if (globaltimer_ns() - t0 > p.timeout_ns) break;
      for (int m = (n > L::kStages ? n - L::kStages : 0); m < n; ++m)
        while (!mbar_try_wait(bar_ring_full(m % L::kStages), (m / L::kStages) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else if (warp == kBwdMmaWarp || warp == kBwdAccWarp) {
    // ======================================================= MMA issuers
    if (lane == 0 && nblk > 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false);
      constexpr uint32_t idAcc = idesc_bf16(128, D, true);
      constexpr uint32_t idDQ = idesc_bf16(128, D, true, true);  // fused dQ: both operands MN-major
      const uint64_t dX = sdesc_kmajor_sw128(sX);
      const uint64_t dX2 = sdesc_kmajor_sw128(sX + L::kTileBytes);
      // S = X·Aᵀ (which = 0) or dP = X2·Bᵀ (which = 1) of block n, all 128
      // columns in one pass over the operands (N = 64 halves would read X
      // from shared memory twice).
      auto product = [&](int n, int which) {
        const uint32_t sT = sRing + (n % L::kStages) * L::kSlotBytes + which * L::kTileBytes;
        const uint64_t dT = sdesc_kmajor_sw128(sT), dXx = which ? dX2 : dX;
        const uint32_t tD = which ? tdP : tS(n);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * L::kSlabBytes + (kk % 4) * 32) >> 4;
          mma_ss(tD, dXx + off, dT + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(which ? bar_dp_full : bar_s_full(n));
      };
      // One half of an accumulation: acc (+)= T[:, 64hh : 64hh+64] · M[64hh : 64hh+64, :]
      // with T packed bf16 in TMEM at tT and M an MN-major tile of block n's slot.
      auto acc_half = [&](int n, int hh, uint32_t tAcc, uint32_t tT, int which) {
        const uint32_t sM = sRing + (n % L::kStages) * L::kSlotBytes + which * L::kTileBytes;
        const uint64_t dM = sdesc_mnmajor_sw128(sM, L::kSlabBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (n > 0 || hh > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tAcc, tT + 8 * kk, dM + (((4 * hh + kk) * 2048) >> 4), idAcc, acc);
        }
      };
      bool ok = true;
      if (warp == kBwdMmaWarp) {
        // ----------------------------------------------- S and dP issuer
        ok = wait_bar(bar_fix, 0, wc) && wait_bar(bar_ring_full(0), 0, wc);
        if (ok) {
          tc_fence_after();
          product(0, 0);
          product(0, 1);
        }
        for (int n = 0; n + 1 < nblk && ok; ++n) {
          if (!wait_bar(bar_ring_full((n + 1) % L::kStages), ((n + 1) / L::kStages) & 1, wc)) { ok = false; break; }
          if (L::kFused) {
            // S(n+1)'s buffer held P(n − 1) and dQ(n − 1), whose read-out
            // follows dV(n − 1); dP(n+1) needs only dP(n) read (dS goes to
            // shared memory).
            if (n >= 1 && !wait_bar(bar_dq_free, (n - 1) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            product(n + 1, 0);
            if (!wait_bar(bar_dp_read, n & 1, wc)) { ok = false; break; }
            tc_fence_after();
            product(n + 1, 1);
          } else if (MODE == kModeDKV) {
            // S(n+1) overwrites P(n): it goes in once dV(n) has completed;
            // dP(n+1) overwrites dS(n) once dK(n) has.
            if (L::kDblS) {  // S(n+1)'s buffer was last read by dV(n − 1)
              if (n >= 1 && !wait_bar(bar_acc_a(n - 1), s_par(n - 1), wc)) { ok = false; break; }
            } else if (!wait_bar(bar_acc_a(n), s_par(n), wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            product(n + 1, 0);
            if (!wait_bar(bar_acc_b, n & 1, wc)) { ok = false; break; }
            tc_fence_after();
            product(n + 1, 1);
          } else {
            // S(n+1) as soon as both warpgroups have read S(n); dP(n+1) as
            // soon as they have read dP(n) (dS has columns of its own).
            for (int hh = 0; hh < 2 && ok; ++hh)
              if (!wait_bar(bar_p_full(hh, n), s_par(n), wc)) ok = false;
            if (!ok) break;
            tc_fence_after();
            product(n + 1, 0);
            if (!wait_bar(bar_dp_read, n & 1, wc)) { ok = false; break; }
            tc_fence_after();
            product(n + 1, 1);
          }
        }
      } else {
        // --------------------------------------------- accumulation issuer
        // The ring slot of block n is released after its last accumulation:
        // S(n) and dP(n), its other readers, have completed by then (the
        // warpgroups stored dS(n) after reading both).
        const uint64_t dDSk = sdesc_kmajor_sw128(sDS);                    // dSᵀ [key, query], K-major
        const uint64_t dDSmn = sdesc_mnmajor_sw128(sDS, L::kSlabBytes);  // dS [query, key], MN-major
        const uint64_t dXmn = sdesc_mnmajor_sw128(sX, L::kSlabBytes);    // K [key, d], MN-major
        for (int n = 0; n < nblk && ok; ++n) {
          if (L::kFused) {
            // dV += Pᵀ dO half by half as the warpgroups store P (TMEM operand).
            for (int hh = 0; hh < 2 && ok; ++hh) {
              if (!wait_bar(bar_p_full(hh, n), s_par(n), wc)) { ok = false; break; }
              tc_fence_after();
              acc_half(n, hh, tAcc0, tS(n) + pcol(hh), 1);
            }
            if (!ok) break;
            mma_commit(bar_acc_a(n));
            // dK += dSᵀ Q half by half as dS lands in shared memory.
            const uint64_t dQt = sdesc_mnmajor_sw128(sRing + (n % L::kStages) * L::kSlotBytes, L::kSlabBytes);
            for (int hh = 0; hh < 2 && ok; ++hh) {
              if (!wait_bar(bar_ds_full(hh, n), ds_par(n), wc)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (n > 0 || hh > 0 || kk > 0) ? 1u : 0u;
                mma_ss(tAcc1, dDSk + ((hh * L::kSlabBytes + kk * 32) >> 4), dQt + (((4 * hh + kk) * 2048) >> 4),
                       idAcc, acc);
              }
            }
            if (!ok) break;
            // dQ(n) = dS K over the block's 128 keys (16 per step).
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tQ(n), dDSmn + ((kk * 2048) >> 4), dXmn + ((kk * 2048) >> 4), idDQ, kk > 0 ? 1u : 0u);
            mma_commit(bar_dq_full);
            mma_commit(bar_ring_empty(n % L::kStages));  // Q(n), dO(n) no longer read
            continue;
          }
          if (MODE == kModeDKV) {
            // dV += Pᵀ dO, half by half as the warpgroups store P.
            for (int hh = 0; hh < 2 && ok; ++hh) {
              if (!wait_bar(bar_p_full(hh, n), s_par(n), wc)) { ok = false; break; }
              tc_fence_after();
              acc_half(n, hh, tAcc0, tS(n) + 64 * hh, 1);
            }
            if (!ok) break;
            mma_commit(bar_acc_a(n));
            // dK += dSᵀ Q.
            for (int hh = 0; hh < 2 && ok; ++hh) {
              if (!wait_bar(bar_ds_full(hh, n), ds_par(n), wc)) { ok = false; break; }
              tc_fence_after();
              acc_half(n, hh, tAcc1, tdP + 64 * hh, 0);
            }
            if (!ok) break;
            mma_commit(bar_acc_b);
          } else {
            // dQ += dS K as the warpgroups store dS.
            for (int hh = 0; hh < 2 && ok; ++hh) {
              if (!wait_bar(bar_ds_full(hh, n), ds_par(n), wc)) { ok = false; break; }
              tc_fence_after();
              acc_half(n, hh, tAcc0, tDS(n) + 32 * hh, 0);
            }
            if (!ok) break;
            mma_commit(bar_dq_done(n & 1));
          }
          mma_commit(bar_ring_empty(n % L::kStages));  // A(n), B(n) no longer read
        }
      }
      // Every MMA must finish before the accumulators are read or TMEM freed
      // (bar_done completes once both issuing threads have committed).
      mma_commit(bar_done);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_done, 0))
        if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else {
    // ============================================ softmax gradient, output
    const int hh = warp >> 2;          // column half
    const int r = threadIdx.x & 127;   // row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int row = r0 + r;            // DQ: query; DKV: key
    // The workspace holds −LSE·log2 e (nl) and D per query; the dQ pass needs
    // its own row's, the dK/dV pass each block's 128 (from the ring slot).
    uint64_t nl_row2 = 0, d_row2 = 0;
    if (MODE == kModeDQ) {
      const float nl = p.lse2[static_cast<size_t>(bh) * p.pitch + row];  // row < n_rt·128 = pitch
      const float dr = p.dvec[static_cast<size_t>(bh) * p.pitch + row];
      nl_row2 = pack2(nl, nl);
      d_row2 = pack2(dr, dr);
    }
    const uint64_t sc2 = pack2(p.scale_log2, p.scale_log2);
    const uint64_t zero2 = 0;
    const bool key_pad = L::kFused && row >= p.Sk;
    // Fused pass: read dQ(m) out of TMEM (which frees its columns), stage it
    // as fp32 with the 128-byte swizzle in the staging buffer, and add it
    // into the fp32 accumulator in device memory, 32 rows × 32 columns per
    // copy.  Warp w owns rows [32(w&3), 32(w&3)+32) and columns
    // [32hh, 32hh+32) of the staging (span hh), and its lane 0 issues their
    // copy; it waits for the copy to have read them only before restaging
    // them for the next block.
    auto dq_out = [&](int m) -> bool {
      const bool got = wait_bar(bar_dq_full, m & 1, wc);
      if (__any_sync(0xffffffffu, !got)) return false;
      tc_fence_after();
      const uint32_t sspan = base + L::kStageOff + hh * (128 * 128);
      if (lane == 0) tma_store_wait_read0();  // the warp's previous copy has read its rows
      __syncwarp();
      uint32_t x[32];
      tmem_ld32(tQ(m) + 32 * hh + lane_off, x);
      tmem_wait_ld();
      reg_fence32(x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_free);
      uint8_t* const rowp = smem + (sspan - base) + r * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(rowp + ((q ^ (r & 7)) << 4)) =
            make_uint4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int qd = warp & 3;
        const int y = (b * p.H + head_of(m)) * p.pitch + col0_of(m) + 32 * qd;
        tma_reduce_add_2d(&tm_dq, sspan + qd * (32 * 128), 32 * hh, y);
        tma_store_commit();
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    for (int n = 0; n < nblk && ok; ++n) {
      const int c0 = col0_of(n);
      const float* vec = reinterpret_cast<const float*>(smem + L::kRingOff + (n % L::kStages) * L::kSlotBytes +
                                                        2 * L::kTileBytes);
      if (L::kKeys) {
        // The block's −log2-LSE and D arrived with its ring slot (which stays
        // loaded until this block's dS has been consumed).
        const bool in = wait_bar(bar_ring_full(n % L::kStages), (n / L::kStages) & 1, wc);
        if (__any_sync(0xffffffffu, !in)) { ok = false; break; }
      }
      // Does any element of this thread's half-block need a mask?
      bool edge;
      if (MODE == kModeDQ) {
        edge = c0 + 64 * hh + 64 > p.Sk || (CAUSAL && c0 + 64 * hh + 63 > r0 + p.coff);
      } else {
        edge = CAUSAL && r0 + 127 > c0 + 64 * hh + p.coff;
      }
      // ---- P = exp2(S·scale·log2 e − LSE₂) over this half's 64 columns
      {
        const bool got = wait_bar(bar_s_full(n), s_par(n), wc);
        if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
      }
      tc_fence_after();
      float pv[64];
      {
        uint32_t us[64];
        tmem_ld32(tS(n) + 64 * hh + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&us[0]));
        tmem_ld32(tS(n) + 64 * hh + 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&us[32]));
        tmem_wait_ld();
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&us[0]));
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&us[32]));
        if (MODE == kModeDQ) {
          // S has been read: its columns may take the next block's S.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_p_full(hh, n));
        }
        uint64_t nlv[32];  // −LSE₂ pairs of this half's columns (dK/dV: 16-byte loads from the slot)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          if (MODE == kModeDQ) {
            nlv[e] = nl_row2;
            nlv[e + 1] = nl_row2;
          } else {
            const uint4 w = *reinterpret_cast<const uint4*>(vec + 64 * hh + 2 * e);
            nlv[e] = (static_cast<uint64_t>(w.y) << 32) | w.x;
            nlv[e + 1] = (static_cast<uint64_t>(w.w) << 32) | w.z;
          }
        }
#pragma unroll
        for (int e = 0; e < 64; e += 2) {  // pairs: x = s·scale·log2 e − LSE₂ (packed fp32)
          const uint64_t nl2 = nlv[e / 2];
          float x0, x1;
          unpack2(ffma2(pack2(__uint_as_float(us[e]), __uint_as_float(us[e + 1])), sc2, nl2), x0, x1);
          float pe[2] = {ex2_mufu(x0), ex2_mufu(x1)};
          if (edge) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int ce = c0 + 64 * hh + e + i;  // global column: DQ key, DKV query
              if (MODE == kModeDQ) {
                if (ce >= p.Sk || (CAUSAL && ce > row + p.coff)) pe[i] = 0.f;
              } else {
                if (CAUSAL && row > ce + p.coff) pe[i] = 0.f;
              }
            }
          }
          pv[e] = pe[0];
          pv[e + 1] = pe[1];
        }
        if (key_pad) {
          // A key row beyond Sk (zero-filled K, V) scores 0, so its P would be
          // exp(−LSE), which overflows for LSE < −88; its dS would then reach
          // dQ as inf · 0.  Such rows contribute nothing.
#pragma unroll
          for (int e = 0; e < 64; ++e) pv[e] = 0.f;
        }
      }
      if (L::kKeys) {
        // Packed bf16 P over 32 of the columns of this half of S.
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
        tmem_st32(tS(n) + pcol(hh) + lane_off, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p_full(hh, n));
      }
      // ---- dS = P ∘ (dP − D)
      {
        const bool got = wait_bar(bar_dp_full, n & 1, wc);
        if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
      }
      tc_fence_after();
      uint32_t qk[32];
      {
        uint32_t ud[64];
        tmem_ld32(tdP + 64 * hh + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&ud[0]));
        tmem_ld32(tdP + 64 * hh + 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&ud[32]));
        tmem_wait_ld();
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&ud[0]));
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&ud[32]));
        if (MODE != kModeDKV) {  // dP(n) is in registers: its columns may take dP(n+1)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dp_read);
        }
#pragma unroll
        for (int e = 0; e < 64; e += 2) {  // pairs: P·(dP − D) (packed fp32)
          uint64_t d2 = d_row2;
          if (L::kKeys) {
            const uint4 w = *reinterpret_cast<const uint4*>(vec + 128 + 64 * hh + (e & ~3));
            d2 = (e & 2) ? ((static_cast<uint64_t>(w.w) << 32) | w.z) : ((static_cast<uint64_t>(w.y) << 32) | w.x);
          }
          const uint64_t diff = fsub2(pack2(__uint_as_float(ud[e]), __uint_as_float(ud[e + 1])), d2);
          float a, b2;
          unpack2(ffma2(pack2(pv[e], pv[e + 1]), diff, zero2), a, b2);
          qk[e / 2] = pack_bf16x2(a, b2);
        }
      }
      if (L::kFused) {
        // The previous block's dQ, computed meanwhile, leaves now.
        if (n >= 1 && !dq_out(n - 1)) {
          ok = false;
          break;
        }
        // dS(n) into row r of slab hh of the shared tile (its readers dK(n − 1)
        // and dQ(n − 1) completed before dQ(n − 1) was read out).
        uint8_t* const rowp = smem + L::kDSOff + hh * L::kSlabBytes + r * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(rowp + ((q ^ (r & 7)) << 4)) =
              make_uint4(qk[4 * q], qk[4 * q + 1], qk[4 * q + 2], qk[4 * q + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ds_full(hh, n));
        continue;
      }
      uint32_t tdst;
      if (MODE == kModeDQ) {
        // dS(n) replaces dS(n−2) in buffer n & 1: dQ(n−2) must have completed
        // (phase (n−2)/2 of that buffer's barrier).
        if (n >= 2) {
          const bool fr = wait_bar(bar_dq_done(n & 1), ((n - 2) >> 1) & 1, wc);
          if (__any_sync(0xffffffffu, !fr)) { ok = false; break; }
          tc_fence_after();
        }
        tdst = tDS(n) + 32 * hh + lane_off;
      } else {
        tdst = tdP + 64 * hh + lane_off;  // over the half of dP this thread has read
      }
      tmem_st32(tdst, qk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds_full(hh, n));
    }
    if (L::kFused && ok && nblk > 0) ok = dq_out(nblk - 1);
    // (shared memory must stay valid until the warp's last copies have read it)
    if (L::kFused && lane == 0) tma_store_wait_read0();
    // ------------------------------------------------------------ outputs
    // The tile's outputs leave by TMA store (rows beyond the tensor are
    // clipped by the copy), staged with the 128-byte swizzle in the X / X2
    // buffers, which are free once the issuer's last commit has completed:
    // every MMA, the last products included, is done then.  Warpgroup hh
    // stages columns [hh·D/2, (hh+1)·D/2) of its rows.
    bool have = nblk > 0 && ok;
    if (have) {
      const bool fin = wait_bar(bar_done, 0, wc);
      if (__any_sync(0xffffffffu, !fin)) have = false;
      tc_fence_after();
    }
    // One decision for all eight warps (they meet at a named barrier below):
    // write the outputs unless a wait anywhere in the CTA ran out.
    uint32_t good;
    {
      const uint32_t mine = ((nblk == 0 || have) && *abort_flag == 0u) ? 1u : 0u;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\t"
          "setp.ne.u32 q, %1, 0;\n\t"
          "bar.red.and.pred p, 1, 256, q;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(good)
          : "r"(mine)
          : "memory");
    }
    if (good) {
      constexpr int kOut = (MODE == kModeDQ) ? 1 : 2;
#pragma unroll
      for (int o = 0; o < kOut; ++o) {
        const uint32_t tacc = (o == 0 ? tAcc0 : tAcc1) + lane_off + hh * (D / 2);
        const float mul = (MODE == kModeDQ || o == 1) ? p.scale : 1.f;
        uint8_t* const stage = smem + L::kXOff + o * L::kTileBytes;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t x[32];
          if (nblk > 0) {
            tmem_ld32(tacc + 32 * c, x);
            tmem_wait_ld();
            reg_fence32(x);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = 0u;  // rows that see no column: zero gradient
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // four 16-byte chunks of 8 values
            uint4 w;
            w.x = pack_bf16x2(mul * __uint_as_float(x[8 * q]), mul * __uint_as_float(x[8 * q + 1]));
            w.y = pack_bf16x2(mul * __uint_as_float(x[8 * q + 2]), mul * __uint_as_float(x[8 * q + 3]));
            w.z = pack_bf16x2(mul * __uint_as_float(x[8 * q + 4]), mul * __uint_as_float(x[8 * q + 5]));
            w.w = pack_bf16x2(mul * __uint_as_float(x[8 * q + 6]), mul * __uint_as_float(x[8 * q + 7]));
            const int col = hh * (D / 2) + 32 * c + 8 * q;
            const int chunk = (col & 63) >> 3;
            *reinterpret_cast<uint4*>(stage + (col >> 6) * L::kSlabBytes + r * 128 + ((chunk ^ (r & 7)) << 4)) = w;
          }
        }
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (threadIdx.x == 0) {
#pragma unroll
        for (int o = 0; o < kOut; ++o)
          for (int sl = 0; sl < L::kSlabs; ++sl)
            tma_store_4d(o == 0 ? &tm_o0 : &tm_o1, sX + o * L::kTileBytes + sl * L::kSlabBytes, 64 * sl, h, r0, b);
        tma_store_commit();
        tma_store_wait_read0();  // shared memory must stay valid until the copy has read it
      }
    }
  }

  // ---- tear-down
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdLoaderWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D = rowsum(dO ∘ O) and −LSE · log2(e) per query row, in [B·H, pitch]
// arrays padded to whole 128-row blocks (−inf and 0 beyond Sq, so padded
// queries get P = 0; negated so that the gradient warps form
// s·scale·log2 e − LSE₂ with one packed FMA per pair).  A warp takes 32·8/D
// rows at once (4 at d = 64, 2 at d = 128): D/8 lanes per row, each reading
// 8 consecutive bf16 of O and of dO as one 16-byte load, and the products are
// summed with shuffles within the row's lanes (O through its element strides
// o_sb, o_ss, o_sh with d contiguous; dO dense).  For the one-pass kernel it
// also zeroes the rows of the dQ accumulator [B·H, pitch, D] (dq_acc
// non-null), 8 fp32 values a lane.
template <int D>
__global__ void attn_bwd_prep_kernel(const uint16_t* o, long long o_sb, long long o_ss, long long o_sh,
                                     const uint16_t* dout, const float* lse, float* lse2, float* dvec, float* dq_acc,
                                     int B, int H, int Sq, int pitch) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, li = lane % kLanesPerRow;
  const long long n = static_cast<long long>(B) * H * pitch;
  const long long groups = (n + kRowsPerWarp - 1) / kRowsPerWarp;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5); g < groups;
       g += warps) {
    const long long t = g * kRowsPerWarp + sub;  // this lane's row
    const bool valid = t < n;
    const int i = static_cast<int>(t % pitch);
    const long long bh = t / pitch;
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
    if (dq_acc != nullptr && valid) {
      float4* const a = reinterpret_cast<float4*>(dq_acc + t * D + 8 * li);
      a[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      a[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc = 0.f;
    if (valid && i < Sq) {
      const size_t off = ((static_cast<size_t>(b) * Sq + i) * H + h) * D + 8 * li;
      const long long ooff = b * o_sb + i * o_ss + h * o_sh + 8 * li;
      const uint4 x = *reinterpret_cast<const uint4*>(o + ooff), y = *reinterpret_cast<const uint4*>(dout + off);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc);
        acc = fmaf(__uint_as_float(xs[e] & 0xFFFF0000u), __uint_as_float(ys[e] & 0xFFFF0000u), acc);
      }
    }
#pragma unroll
    for (int m = kLanesPerRow / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (valid && li == 0) {
      if (i < Sq) {
        dvec[t] = acc;
        lse2[t] = lse[(static_cast<size_t>(b) * H + h) * Sq + i] * -1.4426950408889634f;
      } else {
        lse2[t] = -INFINITY;
        dvec[t] = 0.f;
      }
    }
  }
}

// dQ = scale · (the fused pass's fp32 accumulator), rounded once to bf16:
// acc [B·H, pitch, D] → dq [B, Sq, H, D].  One thread per 8 values (two
// 16-byte loads, one 16-byte store; consecutive threads along the output).
template <int D>
__global__ void attn_bwd_dq_convert_kernel(const float* dq_acc, uint16_t* dq, int B, int H, int Sq, int pitch,
                                           float scale) {
  constexpr int kChunks = D / 8;
  const long long n = static_cast<long long>(B) * Sq * H * kChunks;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(t % kChunks);
    const long long row = t / kChunks;  // (b, i, h) in output order
    const int h = static_cast<int>(row % H);
    const long long bi = row / H;
    const int i = static_cast<int>(bi % Sq);
    const long long bb = bi / Sq;
    const float* src = dq_acc + ((bb * H + h) * pitch + i) * D + 8 * c;
    const float4 lo = *reinterpret_cast<const float4*>(src);
    const float4 hi = *reinterpret_cast<const float4*>(src + 4);
    uint4 w;
    w.x = pack_bf16x2(scale * lo.x, scale * lo.y);
    w.y = pack_bf16x2(scale * lo.z, scale * lo.w);
    w.z = pack_bf16x2(scale * hi.x, scale * hi.y);
    w.w = pack_bf16x2(scale * hi.z, scale * hi.w);
    *reinterpret_cast<uint4*>(dq + row * D + 8 * c) = w;
  }
}

}  // namespace attn

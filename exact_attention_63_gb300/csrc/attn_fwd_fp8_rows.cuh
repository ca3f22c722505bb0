// Exact attention forward with FP8 (E4M3) Q, K and V, head dim 128: full-row
// softmax, two CTAs per SM.
//
// Same operation and method as attn_fwd_fp8_kernel ("FlashAttention-3:
// Pipeline Assíncrono …", section "Estabilidade em FP8": per query tile, a
// first pass over the keys for every row's exact maximum m of the scaled
// logits, then a second for p = 2^(x − m) ≤ 1 and O = P·V with P in E4M3
// under the static scale 448), organised like attn_fwd_rows_kernel:
//
//  * Each CTA takes 256 TMEM columns — S [0, 128) and O [128, 256) — and
//    under half of the shared memory, so two CTAs share every SM and one
//    CTA's exponentials fill the other's waits (pass 1 of one tile beside
//    pass 2 of another).
//  * One softmax warpgroup per CTA; thread r owns query row r (TMEM lane r)
//    and whole 128-key block rows, so the row maximum and the row sum need no
//    exchange between warpgroups.
//  * P8 goes to shared memory as a K-major, 128-byte-swizzled tile (a row of
//    128 E4M3 keys is one swizzle row, the layout of Q), and O += P8·V reads
//    both operands from shared memory.  S is therefore free as soon as the
//    softmax has loaded it: S(g+1) runs while the softmax is still on block g.
//  * Pass 1 does not touch O, so its S blocks alternate between S's columns
//    and O's (once the previous tile's epilogue has read O): S(j+1) of pass 1
//    is computed while the softmax still loads S(j).  A block with no masked
//    key takes its row maximum from the reducing TMEM load (tcgen05.ld.red,
//    the maximum of each 32 columns loaded), not from 64 max instructions.
//  * The factor 448 is folded into the exponent: with m' = m − log2 448,
//    2^(x − m') = 448 p is what E4M3 rounds, the row sum is 448 L, and
//    O = descale_v · (P8·V8) / (448 L), LSE = (m' + log2(448 L)) · ln 2.
//
// Warp roles (256 threads):
//   warp 0     loader (one thread): one K/V ring of 16 KB slots in the order
//              the issuers consume it — per tile, pass 1's K_0 … K_{nb−1},
//              then pass 2's K_0, K_1, V_0, K_2, V_1, … (K two ahead of V);
//              allocates TMEM
//   warp 1     P·V issuer (one thread)
//   warp 2     S issuer (one thread): pass 1 and pass 2 of every tile
//   warp 3     Q loads (two FP8 Q buffers) and output stores (one thread)
//   warps 4-7  softmax, one thread per query row
// Registers: launched at 128 per thread; the role warpgroup gives back to 56
// and the softmax warpgroup takes 200 (setmaxnreg), which holds a row's 128
// scores.  The host launches this kernel only when it was compiled to exactly
// 128 registers, the total both shares add up to.
//
// Output staging: the tile's bf16 output (32 KB) is staged in the tile's Q
// buffer (columns [0, 64)) and the P8 buffer (columns [64, 128)), both free
// once the tile's last P·V has completed; the store warp then loads the Q of
// the tile two ahead into that Q buffer and releases the P8 buffer.
//
// Ordering (every wait is within one phase of the phase it waits for):
//  * S buffer b ∈ {0 (S's columns), 1 (O's columns)}: pass-1 block j uses
//    buffer j & 1, pass 2 buffer 0; issuer and softmax count the uses of each
//    buffer alike.  Use u of buffer b completes s_full[b] and is issued after
//    s_free[b] of use u − 1 (all four softmax warps have loaded it), so
//    s_full[b] cannot run a phase ahead.
//  * Buffer 1's first use in tile t > 0 waits for o_free of tile t − 1 (the
//    epilogue has loaded O); that epilogue needs the whole of tile t − 1, and
//    tile t's first P·V (which overwrites O) needs its pass 1 loaded.
//  * p_full(g'): P8 of pass-2 block g' stored.  P8(g'+1) is stored after
//    pv_done(g'), which needs P·V(g'), issued after p_full(g').
//  * A tile's first P8 is stored after stage_empty of the previous tile (its
//    output store has read the P8 buffer); the store of a tile needs that
//    tile's staging, which comes after its P8 stores.
#pragma once

#include "attn_fwd_fp8.cuh"

namespace attn {

struct Fp8RowsLayout {
  static constexpr int D = 128;
  static constexpr uint32_t kTileBytes = kBM * 128;  // 128 rows × 128 E4M3: one 128-byte-swizzled slab
  static constexpr int kRing = 3;                     // K/V ring slots
  static constexpr uint32_t kQOff = 0;                // two Q buffers (column slab 0 of the output staging)
  static constexpr uint32_t kRingOff = 2 * kTileBytes;
  static constexpr uint32_t kPOff = kRingOff + kRing * kTileBytes;  // P8 (column slab 1 of the output staging)
  static constexpr uint32_t kBarOff = kPOff + kTileBytes;
  // q_full[2], kv_full[R], kv_empty[R], s_full[2], s_free[2], p_full, pv_done, o_final, o_free, stage_full,
  // stage_empty, done[2]
  static constexpr int kNumBars = 2 + 2 * kRing + 4 + 4 + 2 + 2;
  static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;  // tmem base (4 B) + abort flag (4 B)
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS = 0, kColO = 128;
};

constexpr int kFp8RowsThreads = 256;
constexpr int kFp8RowsLaunchRegs = 128;  // 65536 / (2 CTAs × 256 threads)
constexpr int kFp8RowsRoleRegs = 56;
constexpr int kFp8RowsSoftmaxRegs = 200;
static_assert(kFp8RowsThreads / 2 * (kFp8RowsRoleRegs + kFp8RowsSoftmaxRegs) == kFp8RowsThreads * kFp8RowsLaunchRegs,
              "the two register shares must add up to the launch allocation");
// Two CTAs (and the 1 KB the hardware reserves for each) in the SM's 228 KB.
static_assert(2 * (Fp8RowsLayout::kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");

constexpr float kLog2E4M3Max = 8.807354922057604f;  // log2(448)

template <bool CAUSAL>
__global__ void __launch_bounds__(kFp8RowsThreads, 2)
    attn_fwd_fp8_rows_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                             const FwdParams p) {
  using L = Fp8RowsLayout;
  constexpr bool VARLEN = false;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);

  const uint32_t sQ = base + L::kQOff;
  const uint32_t sRing = base + L::kRingOff;
  const uint32_t sP = base + L::kPOff;
  const uint32_t bars = base + L::kBarOff;
  auto bar_q_full = [&](int i) { return bars + 8u * i; };
  auto bar_kv_full = [&](int s) { return bars + 8u * (2 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (2 + L::kRing + s); };
  constexpr uint32_t kB0 = 2 + 2 * L::kRing;
  auto bar_s_full = [&](int b) { return bars + 8u * (kB0 + b); };
  auto bar_s_free = [&](int b) { return bars + 8u * (kB0 + 2 + b); };
  const uint32_t bar_p_full = bars + 8u * (kB0 + 4);
  const uint32_t bar_pv_done = bars + 8u * (kB0 + 5);
  const uint32_t bar_o_final = bars + 8u * (kB0 + 6);
  const uint32_t bar_o_free = bars + 8u * (kB0 + 7);
  const uint32_t bar_stage_full = bars + 8u * (kB0 + 8);
  const uint32_t bar_stage_empty = bars + 8u * (kB0 + 9);
  auto bar_done = [&](int i) { return bars + 8u * (kB0 + 10 + i); };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int stride = static_cast<int>(gridDim.x);
  constexpr int kSmWarps = 4;

  // ---- set-up
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_q_full(i), 1);
      mbar_init(bar_done(i), 1);
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_s_free(i), kSmWarps);
    }
    for (int s = 0; s < L::kRing; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_p_full, kSmWarps);
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_o_final, 1);
    mbar_init(bar_o_free, kSmWarps);
    mbar_init(bar_stage_full, kSmWarps);
    mbar_init(bar_stage_empty, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 2 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const int n_tiles = p.n_tiles;
  // Ring position (relative to the tile's first load) of pass 2's K_j and V_j
  // in a tile of nb blocks; pass 1's K_j sits at j.
  auto pos_k2 = [](int j, int nb) { return nb + (j < 2 ? j : 2 * j - 1); };
  auto pos_v = [](int j, int nb) { return nb + min(2 * j + 2, nb + j); };

  if (warp < 4) {
  // Role warpgroup: give registers back, then one role per warp.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFp8RowsRoleRegs));
  if (warp == 0) {
    // =========================================================== loader
    if (lane == 0) {
      int n = 0;  // ring loads issued
      bool ok = true;
      auto ring_load = [&](const CUtensorMap* m, const Tile& T, int j) -> bool {
        const int slot = n % L::kRing;
        if (!wait_bar(bar_kv_empty(slot), ((n / L::kRing) & 1) ^ 1u, wc)) return false;
        mbar_arrive_expect_tx(bar_kv_full(slot), L::kTileBytes);
        tma_load_4d(sRing + slot * L::kTileBytes, m, 0, T.kvh, j * kBN, T.b, bar_kv_full(slot));
        ++n;
        return true;
      };
      for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride) {
        const Tile T = tile_info<CAUSAL, VARLEN>(idx, p);
        if (p.test_flags & 1u) { ok = false; break; }  // test mode: no K/V copy, the MMA waits must expire
        for (int j = 0; j < T.nb && ok; ++j) ok = ring_load(&tm_k, T, j);  // pass 1
        int kj = 0, vj = 0;                                                // pass 2, K two ahead of V
        while (ok && (kj < T.nb || vj < T.nb)) {
          if (kj < T.nb && kj < vj + 2) ok = ring_load(&tm_k, T, kj++);
          else ok = ring_load(&tm_v, T, vj++);
        }
      }
      const uint64_t t0 = globaltimer_ns();
      for (int i = (n > L::kRing ? n - L::kRing : 0); i < n; ++i)
        while (!mbar_try_wait(bar_kv_full(i % L::kRing), (i / L::kRing) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else if (warp == 3) {
    // ============================================ Q loads, output stores
    if (lane == 0) {
      bool ok = true;
      auto load_q = [&](int idx, int qb) {
        const Tile T = tile_info<CAUSAL, VARLEN>(idx, p);
        mbar_arrive_expect_tx(bar_q_full(qb), L::kTileBytes);
        tma_load_4d(sQ + qb * L::kTileBytes, &tm_q, 0, T.h, T.q0, T.b, bar_q_full(qb));
      };
      int q_issued = 0;
      for (int n = 0; n < 2 && blockIdx.x + n * stride < n_tiles; ++n, ++q_issued)
        load_q(blockIdx.x + n * stride, n);
      int tc = 0;
      for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride, ++tc) {
        const Tile T = tile_info<CAUSAL, VARLEN>(idx, p);
        const int qb = tc & 1;
        if (!wait_bar(bar_stage_full, tc & 1, wc)) { ok = false; break; }
        // Columns [0, 64) are staged in the tile's Q buffer, [64, 128) in the P8 buffer.
        tma_store_4d(&tm_o, sQ + qb * L::kTileBytes, 0, T.h, T.q0, T.b);
        tma_store_4d(&tm_o, sP, 64, T.h, T.q0, T.b);
        tma_store_commit();
        tma_store_wait_read0();
        mbar_arrive(bar_stage_empty);  // the P8 buffer may take the next tile's P8
        if (idx + 2 * stride < n_tiles) {
          load_q(idx + 2 * stride, qb);  // tile tc + 2, into buffer qb
          ++q_issued;
        }
      }
      const uint64_t t0 = globaltimer_ns();
      for (int i = (q_issued > 2 ? q_issued - 2 : 0); i < q_issued; ++i)
        while (!mbar_try_wait(bar_q_full(i & 1), (i >> 1) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else {
    // ====================================================== MMA issuers
    if (lane == 0) {
      bool ok = true;
      if (warp == 2) {
        // ------------------------------------------------------ S issuer
        constexpr uint32_t idS = idesc_e4m3(kBM, kBN, false);
        const uint64_t dQ = sdesc_kmajor_sw128(sQ);
        const uint64_t dK = sdesc_kmajor_sw128(sRing);
        int uses0 = 0, uses1 = 0, tc = 0, tbase = 0;  // uses of S buffer 0 and 1 so far
        for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride, ++tc) {
          const Tile T = tile_info<CAUSAL, VARLEN>(idx, p);
          const int qb = tc & 1;
          if (!wait_bar(bar_q_full(qb), (tc >> 1) & 1, wc)) { ok = false; break; }
          for (int pass = 0; pass < 2 && ok; ++pass) {
            for (int j = 0; j < T.nb; ++j) {
              const int n = tbase + (pass == 0 ? j : pos_k2(j, T.nb)), slot = n % L::kRing;
              const int b = (pass == 0) ? (j & 1) : 0;
              if (!wait_bar(bar_kv_full(slot), (n / L::kRing) & 1, wc)) { ok = false; break; }
              // O's columns take S once the previous tile's epilogue has read O.
              if (b == 1 && j == 1 && tc > 0 && !wait_bar(bar_o_free, (tc - 1) & 1, wc)) { ok = false; break; }
              // The buffer is free once the softmax has loaded its previous S.
              const int u = b ? uses1 : uses0;
              if (u > 0 && !wait_bar(bar_s_free(b), (u - 1) & 1, wc)) { ok = false; break; }
              tc_fence_after();
              const uint64_t dq = dQ + ((qb * L::kTileBytes) >> 4);
              const uint64_t dk = dK + ((slot * L::kTileBytes) >> 4);
              const uint32_t tS = tmem + (b == 0 ? L::kColS : L::kColO);
#pragma unroll
              for (int kk = 0; kk < L::D / 32; ++kk)  // K = 32 E4M3 (32 bytes) per step
                mma_ss_f8(tS, dq + 2 * kk, dk + 2 * kk, idS, kk > 0 ? 1u : 0u);
              mma_commit(bar_s_full(b));
              mma_commit(bar_kv_empty(slot));  // K_j no longer read
              if (b) ++uses1; else ++uses0;
            }
          }
          tbase += 3 * T.nb;
        }
      } else {
        // ---------------------------------------------------- P·V issuer
        constexpr uint32_t idPV = idesc_e4m3(kBM, L::D, true);
        const uint64_t dP = sdesc_kmajor_sw128(sP);
        const uint64_t dV = sdesc_mnmajor_sw128(sRing, L::kTileBytes);
        const uint32_t tO = tmem + L::kColO;
        int gp = 0, tbase = 0;
        for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride) {
          const Tile T = tile_info<CAUSAL, VARLEN>(idx, p);
          for (int j = 0; j < T.nb; ++j, ++gp) {
            const int n = tbase + pos_v(j, T.nb), slot = n % L::kRing;
            if (!wait_bar(bar_kv_full(slot), (n / L::kRing) & 1, wc)) { ok = false; break; }
            if (!wait_bar(bar_p_full, gp & 1, wc)) { ok = false; break; }
            tc_fence_after();
            // O (+)= P8(j) · V_j: four K = 32 steps over the block's 128 keys
            // (A: 32 keys of P8, 32 bytes of each row; B: 32 rows of V, 4 KB).
            const uint64_t dv = dV + ((slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss_f8(tO, dP + 2 * kk, dv + ((kk * 4096) >> 4), idPV, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar_pv_done);
            if (j == T.nb - 1) mma_commit(bar_o_final);
            mma_commit(bar_kv_empty(slot));  // V_j no longer read
          }
          tbase += 3 * T.nb;
        }
      }
      const int me = warp - 1;
      mma_commit(bar_done(me));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_done(me), 0))
        if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  }
  } else {
    // ========================================================== softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kFp8RowsSoftmaxRegs));
    const int r = threadIdx.x & 127;  // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + L::kColO + lane_off;
    const float sc = p.scale_log2;  // scale · descale_q · descale_k · log2(e)
    const uint64_t sc2 = pack2(sc, sc);
    uint8_t* const p_row = smem + L::kPOff + r * 128;  // this row of the P8 tile
    bool ok = true;
    int uses0 = 0, uses1 = 0, gp = 0, tc = 0;  // uses of S buffer 0 and 1 so far
    for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride, ++tc) {
      const Tile T = tile_info<CAUSAL, VARLEN>(idx, p);
      const int q_row = T.q0 + r;
      // Blocks whose keys all lie below Sk and, when causal, at or before the
      // tile's first row need no mask.
      const int lim = CAUSAL ? min(p.Sk, T.q0 + 1 + p.coff) : p.Sk;
      const int n_full = min(T.nb, max(0, lim / kBN));
      // The row's 128 scores of block j (raw logits, fp32) from buffer b,
      // masked; the buffer is released as soon as they are in registers.
      auto load_s = [&](int j, int b, uint32_t (&u)[kBN]) -> bool {
        const bool got = wait_bar_cold(bar_s_full(b), (b ? uses1 : uses0) & 1, wc);
        if (__any_sync(0xffffffffu, !got)) return false;
        tc_fence_after();
        const uint32_t tS = tmem + (b == 0 ? L::kColS : L::kColO) + lane_off;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&u[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32 * c]));
        tc_fence_before();
        warp_arrive(bar_s_free(b), lane);
        if (b) ++uses1; else ++uses0;
        if (j >= n_full) {
          const int k0 = j * kBN;
#pragma unroll
          for (int c = 0; c < kBN; ++c) {
            const int key = k0 + c;
            if (key >= p.Sk || (CAUSAL && key > q_row + p.coff)) u[c] = __float_as_uint(-INFINITY);
          }
        }
        return true;
      };
      // ---------------------------------------------- pass 1: exact maxima
      float m_raw = -INFINITY;
      for (int j = 0; j < T.nb && ok; ++j) {
        uint32_t u[kBN];
        if (j < n_full) {
          // No key of the block is masked: the reducing TMEM load gives each
          // 32 columns' maximum with the values.
          const int b = j & 1;
          const bool got = wait_bar_cold(bar_s_full(b), (b ? uses1 : uses0) & 1, wc);
          if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tS = tmem + (b == 0 ? L::kColS : L::kColO) + lane_off;
          float mc[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld32_max(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&u[32 * c]), mc[c]);
          tmem_wait_ld();
          tc_fence_before();
          warp_arrive(bar_s_free(b), lane);
          if (b) ++uses1; else ++uses0;
          m_raw = fmax3(m_raw, fmax3(mc[0], mc[1], mc[2]), mc[3]);
          continue;
        }
        if (!(ok = load_s(j, j & 1, u))) break;
        const float* const s = reinterpret_cast<const float*>(u);
        float m8[8];  // eight independent 16-wide chains
#pragma unroll
        for (int gg = 0; gg < 8; ++gg) {
          const float* x = s + 16 * gg;
          float a = fmax3(x[0], x[1], x[2]);
          float b2 = fmax3(x[3], x[4], x[5]);
          a = fmax3(a, x[6], x[7]);
          b2 = fmax3(b2, x[8], x[9]);
          a = fmax3(a, x[10], x[11]);
          b2 = fmax3(b2, x[12], x[13]);
          m8[gg] = fmax3(a, b2, fmaxf(x[14], x[15]));
        }
        m_raw = fmax3(m_raw, fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
      }
      if (!ok) break;
      // m' = m − log2 448 (log2 domain), so that 2^(x − m') = 448 p.  Every
      // row sees key 0, so m is finite.
      const float mref = m_raw * sc - kLog2E4M3Max;
      const uint64_t nm2 = pack2(-mref, -mref);
      // --------------------------- pass 2: 448 p = 2^(x − m'), P8 = E4M3(448 p)
      float l_run = 0.f;  // Σ 448 p over the row (unrounded)
      for (int j = 0; j < T.nb && ok; ++j, ++gp) {
        uint32_t u[kBN];
        if (!(ok = load_s(j, 0, u))) break;
        const float* const s = reinterpret_cast<const float*>(u);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t p8[kBN / 4];
#pragma unroll
        for (int i = 0; i < kBN / 4; ++i) {
          float x0, x1, x2, x3;
          unpack2(ffma2(pack2(s[4 * i], s[4 * i + 1]), sc2, nm2), x0, x1);
          unpack2(ffma2(pack2(s[4 * i + 2], s[4 * i + 3]), sc2, nm2), x2, x3);
          x0 = ex2_mufu(x0);
          x1 = ex2_mufu(x1);
          x2 = ex2_mufu(x2);
          x3 = ex2_mufu(x3);
          acc[i & 3] = fadd2(acc[i & 3], fadd2(pack2(x0, x1), pack2(x2, x3)));
          p8[i] = pack_e4m3x4(x0, x1, x2, x3);
        }
        float a0, a1, b0, b1;
        unpack2(fadd2(acc[0], acc[1]), a0, a1);
        unpack2(fadd2(acc[2], acc[3]), b0, b1);
        l_run += (a0 + a1) + (b0 + b1);
        // The P8 buffer is free once the previous P·V has read it and, at a
        // tile's first block, once the previous tile's output store has read
        // its staging there.
        if (gp > 0) {
          const bool landed = wait_bar_cold(bar_pv_done, (gp - 1) & 1, wc);
          if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }
        }
        if (j == 0 && tc > 0) {
          const bool read = wait_bar_cold(bar_stage_empty, (tc - 1) & 1, wc);
          if (__any_sync(0xffffffffu, !read)) { ok = false; break; }
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 8; ++c)  // 16-byte chunk c of the row, 128-byte swizzle
          *reinterpret_cast<uint4*>(p_row + ((c ^ (r & 7)) << 4)) =
              make_uint4(p8[4 * c], p8[4 * c + 1], p8[4 * c + 2], p8[4 * c + 3]);
        fence_proxy_async_smem();  // the MMA reads P8 through the async proxy
        warp_arrive(bar_p_full, lane);
      }
      if (!ok) break;
      // ------------------------------------------------------- epilogue
      // O = descale_v · (P8·V8) / (448 L); staged as bf16, columns [0, 64)
      // in the tile's Q buffer and [64, 128) in the P8 buffer, both free once
      // the tile's last P·V has completed.
      {
        const bool landed = wait_bar(bar_o_final, tc & 1, wc);
        if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }
      }
      tc_fence_after();
      const float f = (l_run > 0.f) ? (p.o_scale * 448.f) / l_run : 0.f;
      const int qb = tc & 1;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t x[32];
        tmem_ld32(tO + 32 * c, x);
        tmem_wait_ld();
        reg_fence32(x);
        uint8_t* const stage = (c < 2) ? smem + L::kQOff + qb * L::kTileBytes : smem + L::kPOff;
#pragma unroll
        for (int q16 = 0; q16 < 4; ++q16) {
          const uint32_t* o8 = &x[8 * q16];
          uint4 wv;
          wv.x = pack_bf16x2(__uint_as_float(o8[0]) * f, __uint_as_float(o8[1]) * f);
          wv.y = pack_bf16x2(__uint_as_float(o8[2]) * f, __uint_as_float(o8[3]) * f);
          wv.z = pack_bf16x2(__uint_as_float(o8[4]) * f, __uint_as_float(o8[5]) * f);
          wv.w = pack_bf16x2(__uint_as_float(o8[6]) * f, __uint_as_float(o8[7]) * f);
          const int chunk = 4 * (c & 1) + q16;  // 16-byte chunk of the slab's 128-byte row
          *reinterpret_cast<uint4*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4)) = wv;
        }
      }
      // O has been read: its columns may take the next tile's pass-1 S.
      tc_fence_before();
      warp_arrive(bar_o_free, lane);
      fence_proxy_async_smem();
      warp_arrive(bar_stage_full, lane);  // the store warp writes the tile out
      if (q_row < p.Sq)
        p.lse[lse0_of<VARLEN>(T, p) + r] = (l_run > 0.f) ? (mref + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
  }

  // ---- tear-down: every role arrives here; all TMEM reads/writes are done
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace attn

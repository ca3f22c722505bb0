// Exact attention forward with FP8 (E4M3) Q, K and V, head dim 128.
//
// "FlashAttention-3: Pipeline Assíncrono …", section "Estabilidade em FP8":
// E4M3 has 3 mantissa bits and a range of ±448, so a one-pass online softmax
// that writes P in FP8 against a running (not yet final) maximum can overflow
// or lose the small terms.  The method takes two passes over each query
// tile's keys: the first computes every row's exact maximum m_i of the scaled
// logits (products accumulated in fp32), the second the exponentials
// p = 2^(x − m_i) ∈ (0, 1] and O = P·V with P in FP8 under a static scale
// (P8 = E4M3(448 p): the row's largest term lands on 448, E4M3's largest
// value).  Q, K and V stand for descale_x · x8 (one scale factor per tensor).
//
// Both products are tcgen05.mma.kind::f8f6f4 (E4M3 × E4M3 → fp32 in TMEM,
// K = 32 per instruction): S = Q·Kᵀ from shared memory (both K-major), and
// O += P·V with P read from TMEM and V (keys × d, MN-major) from shared memory.
//
// Warp roles (384 threads):
//   warp  0    loader: one ring of K/V slots (16 KB each) in the order the
//              issuers consume them — per tile, pass 1's K_0 … K_{nb−1}, then
//              pass 2's K_0, K_1, V_0, K_2, V_1, … (K two ahead of V); every
//              slot is freed by an MMA of an earlier item, so the loader never
//              waits on work that needs a later load.  Allocates TMEM.
//   warp  1    P·V issuer (one thread)
//   warp  2    S issuer (one thread): pass 1 and pass 2 of every tile, S into
//              two TMEM buffers by block parity
//   warp  3    Q loads (two FP8 Q buffers) and output stores (one TMA store
//              per tile from a bf16 staging buffer)
//   warps 4-11 two warpgroups; warpgroup h owns keys [64h, 64h+64) of every
//              block, thread r query row r.  Both halves share the exact
//              maximum, so they feed one O accumulator (no merge, no rescale);
//              they exchange their maxima after pass 1 and their sums at the
//              end of pass 2.
//
// TMEM (512 columns allocated): S buffers [0,128) and [128,256), O [256,384),
// P [384,416) (E4M3, four keys per 32-bit column; half h at 384 + 16h).
//
// Ordering (every parity wait is within one phase of the phase it waits for):
//  * S(g) goes into buffer g & 1 after s_free of block g − 2 (all eight
//    softmax warps have loaded it); s_full(g) then completes.
//  * P(g) is stored after pv_done of the previous pass-2 block (the P buffer's
//    reader); P·V(g) waits for p_full(g).
//  * The tile's Q buffer is released by a commit after its last S (q_empty);
//    the output staging buffer by the store warp once its store has read it
//    (stage_empty).
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

struct Fp8Layout {
  static constexpr int D = 128;
  static constexpr uint32_t kTileBytes = kBM * 128;  // 128 rows × 128 E4M3 = one 128-byte-swizzled slab
  static constexpr int kRing = 6;                     // K/V ring slots
  static constexpr uint32_t kQOff = 0;                // two Q buffers
  static constexpr uint32_t kRingOff = 2 * kTileBytes;
  static constexpr uint32_t kStageOff = kRingOff + kRing * kTileBytes;  // bf16 O: two 16 KB slabs
  static constexpr uint32_t kStageBytes = 2 * kBM * 128;
  // per-row maxima and sums of each half, double-buffered by tile parity: [2][2][128] float each
  static constexpr uint32_t kStatsOff = kStageOff + kStageBytes;
  static constexpr uint32_t kStatsBytes = 2 * 2 * 2 * kBM * 4;
  static constexpr uint32_t kBarOff = kStatsOff + kStatsBytes;
  // q_full[2], q_empty[2], kv_full[R], kv_empty[R], s_full[2], s_free[2], p_full, pv_done, o_final,
  // xm_full, xl_full, stage_full, stage_empty, done[2]
  static constexpr int kNumBars = 4 + 2 * kRing + 4 + 3 + 4 + 2;
  static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;  // tmem base (4 B) + abort flag (4 B)
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
};

// Four fp32 values → four E4M3 bytes (round to nearest even, saturating),
// x0 in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4: E4M3 × E4M3 → fp32,
// A K-major, B K-major (b_mn = false) or MN-major (b_mn = true).
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool b_mn) {
  return (1u << 4)                                 // accumulator fp32
         | (0u << 7)                               // A E4M3
         | (0u << 10)                              // B E4M3
         | ((b_mn ? 1u : 0u) << 16)                // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// D[tmem] (+)= A[smem] · B[smem], FP8 operands
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] · B[smem], FP8 operands
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const FwdParams p) {
  using L = Fp8Layout;
  constexpr bool VARLEN = false;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);

  const uint32_t sQ = base + L::kQOff;
  const uint32_t sRing = base + L::kRingOff;
  const uint32_t sStage = base + L::kStageOff;
  const uint32_t bars = base + L::kBarOff;
  auto bar_q_full = [&](int i) { return bars + 8u * i; };
  auto bar_q_empty = [&](int i) { return bars + 8u * (2 + i); };
  auto bar_kv_full = [&](int s) { return bars + 8u * (4 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (4 + L::kRing + s); };
  constexpr uint32_t kB0 = 4 + 2 * L::kRing;
  auto bar_s_full = [&](int i) { return bars + 8u * (kB0 + i); };
  auto bar_s_free = [&](int i) { return bars + 8u * (kB0 + 2 + i); };
  const uint32_t bar_p_full = bars + 8u * (kB0 + 4);
  const uint32_t bar_pv_done = bars + 8u * (kB0 + 5);
  const uint32_t bar_o_final = bars + 8u * (kB0 + 6);
  const uint32_t bar_xm_full = bars + 8u * (kB0 + 7);
  const uint32_t bar_xl_full = bars + 8u * (kB0 + 8);
  const uint32_t bar_stage_full = bars + 8u * (kB0 + 9);
  const uint32_t bar_stage_empty = bars + 8u * (kB0 + 10);
  auto bar_done = [&](int i) { return bars + 8u * (kB0 + 11 + i); };
  float* const stats = reinterpret_cast<float*>(smem + L::kStatsOff);  // [tile parity][m / l][half][row]
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int stride = static_cast<int>(gridDim.x);
  constexpr int kSmWarps = 8;

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
      mbar_init(bar_q_empty(i), 1);
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_s_free(i), kSmWarps);
      mbar_init(bar_done(i), 1);
    }
    for (int s = 0; s < L::kRing; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_p_full, kSmWarps);
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_o_final, 1);
    mbar_init(bar_xm_full, kSmWarps);
    mbar_init(bar_xl_full, kSmWarps);
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
  const int* const seq_tab = nullptr;
  // Ring position (relative to the tile's first load) of pass 2's K_j and V_j
  // in a tile of nb blocks; pass 1's K_j sits at j.
  auto pos_k2 = [](int j, int nb) { return nb + (j < 2 ? j : 2 * j - 1); };
  auto pos_v = [](int j, int nb) { return nb + min(2 * j + 2, nb + j); };

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
        const Tile T = tile_info<CAUSAL, VARLEN>(idx, p, seq_tab);
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
      auto load_q = [&](const Tile& T, int qb) {
        mbar_arrive_expect_tx(bar_q_full(qb), L::kTileBytes);
        tma_load_4d(sQ + qb * L::kTileBytes, &tm_q, 0, T.h, T.q0, T.b, bar_q_full(qb));
      };
      int q_issued = 0;
      for (int idx = blockIdx.x, n = 0; idx < n_tiles && n < 2; idx += stride, ++n, ++q_issued)
        load_q(tile_info<CAUSAL, VARLEN>(idx, p, seq_tab), n);
      int tc = 0;
      for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride, ++tc) {
        const Tile T = tile_info<CAUSAL, VARLEN>(idx, p, seq_tab);
        const int qb = tc & 1;
        // Tile tc's Q buffer takes tile tc + 2's Q once its last S completed.
        if (idx + 2 * stride < n_tiles) {
          if (!wait_bar(bar_q_empty(qb), (tc >> 1) & 1, wc)) { ok = false; break; }
          load_q(tile_info<CAUSAL, VARLEN>(idx + 2 * stride, p, seq_tab), qb);
          ++q_issued;
        }
        if (!wait_bar(bar_stage_full, tc & 1, wc)) { ok = false; break; }
        for (int sl = 0; sl < 2; ++sl)
          tma_store_4d(&tm_o, sStage + sl * (kBM * 128), 64 * sl, T.h, T.q0, T.b);
        tma_store_commit();
        tma_store_wait_read0();
        mbar_arrive(bar_stage_empty);
      }
      const uint64_t t0 = globaltimer_ns();
      for (int i = (q_issued > 2 ? q_issued - 2 : 0); i < q_issued; ++i)
        while (!mbar_try_wait(bar_q_full(i & 1), (i >> 1) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else if (warp == 1 || warp == 2) {
    // ====================================================== MMA issuers
    if (lane == 0) {
      bool ok = true;
      if (warp == 2) {
        // ------------------------------------------------------ S issuer
        constexpr uint32_t idS = idesc_e4m3(kBM, kBN, false);
        const uint64_t dQ = sdesc_kmajor_sw128(sQ);
        const uint64_t dK = sdesc_kmajor_sw128(sRing);
        int gs = 0, tc = 0, tbase = 0;
        for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride, ++tc) {
          const Tile T = tile_info<CAUSAL, VARLEN>(idx, p, seq_tab);
          const int qb = tc & 1;
          if (!wait_bar(bar_q_full(qb), (tc >> 1) & 1, wc)) { ok = false; break; }
          for (int pass = 0; pass < 2 && ok; ++pass) {
            for (int j = 0; j < T.nb; ++j, ++gs) {
              const int buf = gs & 1;
              const int n = tbase + (pass == 0 ? j : pos_k2(j, T.nb)), slot = n % L::kRing;
              if (!wait_bar(bar_kv_full(slot), (n / L::kRing) & 1, wc)) { ok = false; break; }
              if (gs >= 2 && !wait_bar(bar_s_free(buf), ((gs - 2) >> 1) & 1, wc)) { ok = false; break; }
              tc_fence_after();
              const uint64_t dq = dQ + ((qb * L::kTileBytes) >> 4);
              const uint64_t dk = dK + ((slot * L::kTileBytes) >> 4);
              const uint32_t tS = tmem + L::kColS + 128u * buf;
#pragma unroll
              for (int kk = 0; kk < L::D / 32; ++kk)  // K = 32 E4M3 (32 bytes) per step
                mma_ss_f8(tS, dq + 2 * kk, dk + 2 * kk, idS, kk > 0 ? 1u : 0u);
              mma_commit(bar_s_full(buf));
              mma_commit(bar_kv_empty(slot));  // K_j no longer read
              if (pass == 1 && j == T.nb - 1) mma_commit(bar_q_empty(qb));  // the tile's Q no longer read
            }
          }
          tbase += 3 * T.nb;
        }
      } else {
        // ---------------------------------------------------- P·V issuer
        constexpr uint32_t idPV = idesc_e4m3(kBM, L::D, true);
        const uint64_t dV = sdesc_mnmajor_sw128(sRing, L::kTileBytes);
        const uint32_t tP = tmem + L::kColP;
        const uint32_t tO = tmem + L::kColO;
        int gp = 0, tbase = 0;
        for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride) {
          const Tile T = tile_info<CAUSAL, VARLEN>(idx, p, seq_tab);
          for (int j = 0; j < T.nb; ++j, ++gp) {
            const int n = tbase + pos_v(j, T.nb), slot = n % L::kRing;
            if (!wait_bar(bar_kv_full(slot), (n / L::kRing) & 1, wc)) { ok = false; break; }
            if (!wait_bar(bar_p_full, gp & 1, wc)) { ok = false; break; }
            tc_fence_after();
            // O (+)= P(j) · V_j: four K = 32 steps over the block's 128 keys
            // (A: 8 TMEM columns of four E4M3 each; B: 32 rows of V, 4 KB).
            const uint64_t dv = dV + ((slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts_f8(tO, tP + kk * 8, dv + ((kk * 4096) >> 4), idPV, (j > 0 || kk > 0) ? 1u : 0u);
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
  } else {
    // ========================================================== softmax
    const int h = (warp - 4) >> 2;    // key half owned by this warpgroup
    const int r = threadIdx.x & 127;  // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sc = p.scale_log2;    // scale · descale_q · descale_k · log2(e)
    const uint64_t sc2 = pack2(sc, sc);
    constexpr int kHalf = kBN / 2;
    bool ok = true;
    int gs = 0, gp = 0, tc = 0;
    for (int idx = blockIdx.x; idx < n_tiles && ok; idx += stride, ++tc) {
      const Tile T = tile_info<CAUSAL, VARLEN>(idx, p, seq_tab);
      const int q_row = T.q0 + r;
      const int lim = CAUSAL ? min(p.Sk, T.q0 + 1 + p.coff) : p.Sk;
      // Blocks whose keys of this half all lie below lim need no mask.
      const int n_full = min(T.nb, max(0, (lim - kHalf * h + kHalf) / kBN));
      // This half's 64 scores of block gs (raw logits, fp32), masked.
      auto load_s = [&](int j, float (&s)[kHalf]) -> bool {
        const int buf = gs & 1;
        const bool got = wait_bar_cold(bar_s_full(buf), (gs >> 1) & 1, wc);
        if (__any_sync(0xffffffffu, !got)) return false;
        tc_fence_after();
        uint32_t* const u = reinterpret_cast<uint32_t*>(s);
        const uint32_t tS = tmem + L::kColS + 128u * buf + kHalf * h + lane_off;
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tmem_wait_ld();
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tc_fence_before();
        warp_arrive(bar_s_free(buf), lane);  // S(gs) is in registers
        if (j >= n_full) {
          const int k0 = j * kBN + kHalf * h;
#pragma unroll
          for (int c = 0; c < kHalf; ++c) {
            const int key = k0 + c;
            if (key >= p.Sk || (CAUSAL && key > q_row + p.coff)) s[c] = -INFINITY;
          }
        }
        return true;
      };
      // ---------------------------------------------- pass 1: exact maxima
      float m_h = -INFINITY;
      for (int j = 0; j < T.nb && ok; ++j, ++gs) {
        float s[kHalf];
        if (!(ok = load_s(j, s))) break;
        float m4[4];
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const float* x = s + 16 * gg;
          float a = fmax3(x[0], x[1], x[2]);
          float b2 = fmax3(x[3], x[4], x[5]);
          a = fmax3(a, x[6], x[7]);
          b2 = fmax3(b2, x[8], x[9]);
          a = fmax3(a, x[10], x[11]);
          b2 = fmax3(b2, x[12], x[13]);
          m4[gg] = fmax3(a, b2, fmaxf(x[14], x[15]));
        }
        m_h = fmax3(m_h, fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      if (!ok) break;
      float* const st = stats + (tc & 1) * (2 * 2 * kBM);
      st[h * kBM + r] = m_h;
      warp_arrive(bar_xm_full, lane);
      {
        const bool in = wait_bar(bar_xm_full, tc & 1, wc);
        if (__any_sync(0xffffffffu, !in)) { ok = false; break; }
      }
      // The row's exact maximum of the scaled logits (log2 domain).  Every
      // row sees key 0, so it is finite.
      const float m = fmaxf(st[r], st[kBM + r]) * sc;
      const uint64_t nm2 = pack2(-m, -m);
      // ----------------------- pass 2: p = 2^(x − m) ≤ 1, P8 = E4M3(448 p)
      float l_h = 0.f;
      for (int j = 0; j < T.nb && ok; ++j, ++gs, ++gp) {
        float s[kHalf];
        if (!(ok = load_s(j, s))) break;
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t p8[kHalf / 4];
#pragma unroll
        for (int i = 0; i < kHalf / 4; ++i) {
          float x0, x1, x2, x3;
          unpack2(ffma2(pack2(s[4 * i], s[4 * i + 1]), sc2, nm2), x0, x1);
          unpack2(ffma2(pack2(s[4 * i + 2], s[4 * i + 3]), sc2, nm2), x2, x3);
          x0 = ex2_mufu(x0);
          x1 = ex2_mufu(x1);
          x2 = ex2_mufu(x2);
          x3 = ex2_mufu(x3);
          acc[i & 3] = fadd2(acc[i & 3], fadd2(pack2(x0, x1), pack2(x2, x3)));
          p8[i] = pack_e4m3x4(448.f * x0, 448.f * x1, 448.f * x2, 448.f * x3);
        }
        float a0, a1, b0, b1;
        unpack2(fadd2(acc[0], acc[1]), a0, a1);
        unpack2(fadd2(acc[2], acc[3]), b0, b1);
        l_h += (a0 + a1) + (b0 + b1);
        // The P buffer is free once the previous P·V has read it.
        if (gp > 0) {
          const bool landed = wait_bar_cold(bar_pv_done, (gp - 1) & 1, wc);
          if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st16(tmem + L::kColP + 16 * h + lane_off, p8);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar_p_full, lane);
      }
      if (!ok) break;
      // ------------------------------------------------------- epilogue
      st[2 * kBM + h * kBM + r] = l_h;
      warp_arrive(bar_xl_full, lane);
      {
        const bool in = wait_bar(bar_xl_full, tc & 1, wc);
        if (__any_sync(0xffffffffu, !in)) { ok = false; break; }
      }
      const float Lsum = st[2 * kBM + r] + st[3 * kBM + r];
      // O = descale_v · (P8 · V8) / (448 · L); warpgroup h writes columns [64h, 64h+64).
      const float f = (Lsum > 0.f) ? p.o_scale / Lsum : 0.f;
      {
        const bool landed = wait_bar(bar_o_final, tc & 1, wc);
        if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }
      }
      if (tc > 0) {  // the staging buffer is free once the previous tile's store has read it
        const bool free_ = wait_bar(bar_stage_empty, (tc - 1) & 1, wc);
        if (__any_sync(0xffffffffu, !free_)) { ok = false; break; }
      }
      tc_fence_after();
      uint8_t* const stage = smem + L::kStageOff + h * (kBM * 128);  // slab h holds columns [64h, 64h+64)
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t x[32];
        tmem_ld32(tmem + L::kColO + 64 * h + 32 * c + lane_off, x);
        tmem_wait_ld();
        reg_fence32(x);
#pragma unroll
        for (int q16 = 0; q16 < 4; ++q16) {
          const uint32_t* o8 = &x[8 * q16];
          uint4 wv;
          wv.x = pack_bf16x2(__uint_as_float(o8[0]) * f, __uint_as_float(o8[1]) * f);
          wv.y = pack_bf16x2(__uint_as_float(o8[2]) * f, __uint_as_float(o8[3]) * f);
          wv.z = pack_bf16x2(__uint_as_float(o8[4]) * f, __uint_as_float(o8[5]) * f);
          wv.w = pack_bf16x2(__uint_as_float(o8[6]) * f, __uint_as_float(o8[7]) * f);
          const int chunk = 4 * c + q16;  // 16-byte chunk of the slab's 128-byte row
          *reinterpret_cast<uint4*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4)) = wv;
        }
      }
      fence_proxy_async_smem();
      warp_arrive(bar_stage_full, lane);
      if (h == 0 && q_row < p.Sq)
        p.lse[lse0_of<VARLEN>(T, p) + r] = (Lsum > 0.f) ? (m + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
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

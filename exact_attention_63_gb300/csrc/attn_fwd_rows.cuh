// Exact attention forward for head dim 64: full-row softmax, two CTAs per SM.
//
// Same operation, tiles and parameters as attn_fwd_kernel (one tile = 128
// query rows of one (batch, head) against every visible 128-key block, online
// softmax, O and LSE out; "FlashAttention 4: Atenção Mais Rápida …", section
// "Novidades no FlashAttention 4"), organised for d = 64, where a block holds
// half the tensor work of d = 128 per exponential and the per-block hand-offs
// between the softmax and the MMA issuers, not the tensor core, set the pace:
//
//  * Each CTA takes 256 of the SM's 512 TMEM columns and under half of its
//    shared memory, so two CTAs share every SM.  Their pipelines are
//    independent: each has its own S and P·V issuing threads (one thread
//    issues at most one tcgen05.mma per ~45 cycles, a 128×64×16 P·V step
//    takes the tensor core 32), and one CTA's exponentials fill the other's
//    barrier waits on the schedulers and the MUFU pipe.
//  * One softmax warpgroup per CTA; thread r owns query row r (TMEM lane r)
//    and the whole 128-key block row, so there is one running maximum, row
//    sum and O accumulator per row and no merge of halves.
//  * P has TMEM columns of its own, so the S buffer is free as soon as the
//    softmax has loaded S(j) into registers: S(j+1) = Q·K_{j+1}ᵀ runs while
//    the softmax is still on block j.  P(j+1) is stored once P(j)·V (the P
//    buffer's reader) has completed.
//
// Warp roles (256 threads):
//   warp 0     loader (one thread): K/V ring of 3 slots in consumption order
//              K_0, K_1, then V_g, K_{g+2} per block g; allocates TMEM
//   warp 1     P·V issuer (one thread): O += P(j) · V_j, P from TMEM
//   warp 2     S issuer (one thread): S = Q · K_jᵀ
//   warp 3     Q loads and output stores (one thread), as in attn_fwd_kernel
//   warps 4-7  softmax, one thread per query row
// Registers: launched at 128 per thread; the role warpgroup gives back to 56
// and the softmax warpgroup takes 200 (setmaxnreg), which holds a row's 128
// scores in registers while it computes the exponentials.  The host launches this kernel only when it was
// compiled to exactly 128 registers, the total both shares add up to.
//
// TMEM columns (256): S [0, 128), P [128, 192) (bf16 pairs), O [192, 256).
//
// Ordering (every wait is within one phase of the phase it waits for):
//  * s_full(j): S(j) complete.  S(j+1) is issued after s_free(j) (all four
//    softmax warps have loaded S(j)), so s_full cannot run a phase ahead.
//  * p_full(j): P(j) stored.  P(j+1) is stored after pv_done(j), which needs
//    P·V(j), issued after p_full(j).
//  * O is rescaled at block j only after pv_done(j−1) and before p_full(j),
//    and P·V(j) waits for p_full(j); the epilogue reads O after o_final (the
//    tile's last P·V), before the next tile's first p_full.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

struct RowsLayout {
  static constexpr int D = 64;
  static constexpr uint32_t kTileBytes = kBM * 128;  // 128 rows × 64 bf16: one 128-byte-swizzled slab
  static constexpr int kStages = 3;                   // K/V ring slots
  static constexpr int kLook = 2;                     // K runs this many blocks ahead of V in the ring order
  static constexpr uint32_t kQOff = 0;                // two Q buffers (also the output staging)
  static constexpr uint32_t kRingOff = 2 * kTileBytes;
  static constexpr uint32_t kBarOff = kRingOff + kStages * kTileBytes;
  // q_full[2], kv_full[S], kv_empty[S], s_full, s_free, p_full, pv_done, o_final, stage_full[2], done[2]
  static constexpr int kNumBars = 2 + 2 * kStages + 5 + 2 + 2;
  static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;  // tmem base (4 B) + abort flag (4 B)
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base to 1024
  // Packed sequences without a causal mask: the sequence tile table and its
  // scratch (one int per warp) after the words, in extra shared memory.
  static constexpr uint32_t kTableOff = kMiscOff + 16;
  static constexpr uint32_t kSmemBytesTable = kSmemBytes + kSeqTableBytes + 64;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;
};

constexpr int kRowsThreads = 256;
constexpr int kRowsLaunchRegs = 128;  // 65536 / (2 CTAs × 256 threads)
constexpr int kRowsRoleRegs = 56;
constexpr int kRowsSoftmaxRegs = 200;  // 128·56 + 128·200 = 256·128
static_assert(kRowsThreads / 2 * (kRowsRoleRegs + kRowsSoftmaxRegs) == kRowsThreads * kRowsLaunchRegs,
              "the two register shares must add up to the launch allocation");

// POLY: bit c selects the FMA-pipe polynomial exp2 for 16-key chunk c of
// every 128-key block (compile time, so the exp loop is one basic block).
// VARLEN: sequences of different lengths packed along the rows, as in
// attn_fwd_kernel (a sequence's last tile written row by row, rows that see
// no key set to O = 0, LSE = −inf).
template <bool CAUSAL, bool COUNT, uint32_t POLY, bool VARLEN>
__global__ void __launch_bounds__(kRowsThreads, 2)
    attn_fwd_rows_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const FwdParams p) {
  using L = RowsLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);

  const uint32_t sQ = base + L::kQOff;
  const uint32_t sRing = base + L::kRingOff;
  const uint32_t bars = base + L::kBarOff;
  auto bar_q_full = [&](int i) { return bars + 8u * i; };
  auto bar_kv_full = [&](int s) { return bars + 8u * (2 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (2 + L::kStages + s); };
  constexpr uint32_t kB0 = 2 + 2 * L::kStages;
  const uint32_t bar_s_full = bars + 8u * kB0;
  const uint32_t bar_s_free = bars + 8u * (kB0 + 1);
  const uint32_t bar_p_full = bars + 8u * (kB0 + 2);
  const uint32_t bar_pv_done = bars + 8u * (kB0 + 3);
  const uint32_t bar_o_final = bars + 8u * (kB0 + 4);
  auto bar_stage_full = [&](int i) { return bars + 8u * (kB0 + 5 + i); };
  auto bar_done = [&](int i) { return bars + 8u * (kB0 + 7 + i); };
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
      mbar_init(bar_stage_full(i), kSmWarps);
      mbar_init(bar_done(i), 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_free, kSmWarps);
    mbar_init(bar_p_full, kSmWarps);
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_o_final, 1);
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
  int n_tiles = p.n_tiles;
  const int* seq_tab = nullptr;
  if constexpr (VARLEN && !CAUSAL) {  // the tiles that hold rows, in order (every thread takes part)
    if (p.B <= kSeqTableCap) {
      int* const tab = reinterpret_cast<int*>(smem + L::kTableOff);
      n_tiles = build_seq_table(p, tab, tab + kSeqTableCap + 1);
      seq_tab = tab;
    }
  }

  if (warp < 4) {
  // Role warpgroup: give registers back, then one role per warp.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRowsRoleRegs));
  if (warp == 0) {
    // =========================================================== loader
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      Tile k_T, v_T;
      int k_idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, k_T, n_tiles, seq_tab), k_j = 0, gK = 0;
      int v_idx = k_idx, v_j = 0, gV = 0;
      v_T = k_T;
      auto ring_load = [&](const CUtensorMap* m, const Tile& T, int j) -> bool {
        const int slot = issued % L::kStages;
        if (!wait_bar(bar_kv_empty(slot), ((issued / L::kStages) & 1) ^ 1u, wc)) return false;
        mbar_arrive_expect_tx(bar_kv_full(slot), L::kTileBytes);
        tma_load_4d(sRing + slot * L::kTileBytes, m, 0, T.kvh, krow_of<VARLEN>(T) + j * kBN, bcoord_of<VARLEN>(T),
                    bar_kv_full(slot));
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
      while (ok && k_idx < n_tiles && gK < gV + L::kLook) ok = load_k();
      while (ok && v_idx < n_tiles) {
        if (!ring_load(&tm_v, v_T, v_j)) { ok = false; break; }
        ++gV;
        if (++v_j == v_T.nb) {
          v_j = 0;
          v_idx = next_running<CAUSAL, VARLEN>(v_idx + stride, stride, p, v_T, n_tiles, seq_tab);
        }
        while (ok && k_idx < n_tiles && gK < gV + L::kLook) ok = load_k();
      }
      const uint64_t t0 = globaltimer_ns();
      for (int n = (issued > L::kStages ? issued - L::kStages : 0); n < issued; ++n)
        while (!mbar_try_wait(bar_kv_full(n % L::kStages), (n / L::kStages) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else if (warp == 3) {
    // ===================================================== output store
    // As in attn_fwd_kernel: the softmax warps stage each tile's bf16 output
    // in the tile's Q buffer; one TMA store writes it, then the Q of the tile
    // two ahead is loaded into that buffer.
    if (lane == 0) {
      Tile Tq;
      int q_idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, Tq, n_tiles, seq_tab), q_issued = 0;
      auto load_q = [&]() {
        const int qb = q_issued & 1;
        mbar_arrive_expect_tx(bar_q_full(qb), L::kTileBytes);
        tma_load_4d(sQ + qb * L::kTileBytes, &tm_q, 0, Tq.h, qrow_of<VARLEN>(Tq), bcoord_of<VARLEN>(Tq),
                    bar_q_full(qb));
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
          tma_store_4d(&tm_o, sQ + qb * L::kTileBytes, 0, T.h, qrow_of<VARLEN>(T), bcoord_of<VARLEN>(T));
          tma_store_commit();
          tma_store_wait_read0();
        }
        if (q_idx < n_tiles) load_q();  // tile tc + 2, into buffer qb
      }
      const uint64_t t0 = globaltimer_ns();
      for (int n = (q_issued > 2 ? q_issued - 2 : 0); n < q_issued; ++n)
        while (!mbar_try_wait(bar_q_full(n & 1), (n >> 1) & 1u))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else if (warp == 1 || warp == 2) {
    // ====================================================== MMA issuers
    // Ring positions (loader's order): K_j → j for j < kLook, else
    // 2j − kLook + 1; V_g → min(2g + kLook, G + g) over the CTA's G blocks.
    if (lane == 0) {
      bool ok = true;
      if (warp == 2) {
        // ------------------------------------------------------ S issuer
        constexpr uint32_t idS = idesc_bf16(kBM, kBN, false);
        const uint64_t dQ = sdesc_kmajor_sw128(sQ);
        const uint64_t dK = sdesc_kmajor_sw128(sRing);
        const uint32_t tS = tmem + L::kColS;
        int g = 0, tc = 0;
        Tile T;
        for (int idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, T, n_tiles, seq_tab); idx < n_tiles && ok;
             idx = next_running<CAUSAL, VARLEN>(idx + stride, stride, p, T, n_tiles, seq_tab), ++tc) {
          const int qb = tc & 1;
          for (int j = 0; j < T.nb; ++j, ++g) {
            if (j == 0 && !wait_bar(bar_q_full(qb), (tc >> 1) & 1, wc)) { ok = false; break; }
            const int n = (g < L::kLook) ? g : 2 * g - L::kLook + 1, slot = n % L::kStages;
            if (!wait_bar(bar_kv_full(slot), (n / L::kStages) & 1, wc)) { ok = false; break; }
            // The S buffer is free once the softmax has loaded S(g−1).
            if (g > 0 && !wait_bar(bar_s_free, (g - 1) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dq = dQ + ((qb * L::kTileBytes) >> 4);
            const uint64_t dk = dK + ((slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < L::D / 16; ++kk) mma_ss(tS, dq + 2 * kk, dk + 2 * kk, idS, kk > 0 ? 1u : 0u);
            mma_commit(bar_s_full);
            mma_commit(bar_kv_empty(slot));  // K_j no longer read
          }
        }
      } else {
        // ---------------------------------------------------- P·V issuer
        constexpr uint32_t idPV = idesc_bf16(kBM, L::D, true);
        const uint64_t dV = sdesc_mnmajor_sw128(sRing, L::kTileBytes);
        const uint32_t tP = tmem + L::kColP;
        const uint32_t tO = tmem + L::kColO;
        Tile T;
        int G = 0;
        for (int idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, T, n_tiles, seq_tab); idx < n_tiles;
             idx = next_running<CAUSAL, VARLEN>(idx + stride, stride, p, T, n_tiles, seq_tab))
          G += T.nb;
        int g = 0;
        for (int idx = next_running<CAUSAL, VARLEN>(blockIdx.x, stride, p, T, n_tiles, seq_tab); idx < n_tiles && ok;
             idx = next_running<CAUSAL, VARLEN>(idx + stride, stride, p, T, n_tiles, seq_tab)) {
          for (int j = 0; j < T.nb; ++j, ++g) {
            const int n = min(2 * g + L::kLook, G + g), slot = n % L::kStages;
            if (!wait_bar(bar_kv_full(slot), (n / L::kStages) & 1, wc)) { ok = false; break; }
            if (!wait_bar(bar_p_full, g & 1, wc)) { ok = false; break; }
            tc_fence_after();
            // O (+)= P(g) · V_j: eight K = 16 steps over the block's 128 keys
            // (A: 8 TMEM columns of bf16 pairs each; B: 16 rows of V, 2 KB).
            const uint64_t dv = dV + ((slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tO, tP + kk * 8, dv + ((kk * 2048) >> 4), idPV, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar_pv_done);
            if (j == T.nb - 1) mma_commit(bar_o_final);
            mma_commit(bar_kv_empty(slot));  // V_j no longer read
          }
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRowsSoftmaxRegs));
    const int r = threadIdx.x & 127;  // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + L::kColS + lane_off;
    const uint32_t tP = tmem + L::kColP + lane_off;
    const uint32_t tO = tmem + L::kColO + lane_off;
    const float sc = p.scale_log2;
    const uint64_t sc2 = pack2(sc, sc);
    bool ok = true;
    int g = 0, tc = 0;
    bool s_ready = false;  // S(g) known complete (tested at the end of block g − 1)
    // O row of this thread in tile T (element offset), for the rows the
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
            uint4* const dst = reinterpret_cast<uint4*>(o_row(T));
#pragma unroll
            for (int c = 0; c < L::D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[T.lse0 + r] = -INFINITY;
          }
          continue;
        }
      }
      float m_run = -INFINITY;  // running reference maximum (log2 domain)
      float l_run = 0.f;        // running row sum (fp32, unrounded p)
      auto block = [&](int j, auto mask_tag) -> bool {
        constexpr bool MASK = decltype(mask_tag)::value;
        const bool got = s_ready || wait_bar_cold(bar_s_full, g & 1, wc);
        if (__any_sync(0xffffffffu, !got)) return false;
        tc_fence_after();
        uint32_t u[kBN];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&u[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32 * c]));
        // S(g) is in registers: the S buffer is free for S(g+1).
        tc_fence_before();
        warp_arrive(bar_s_free, lane);
        float* const s = reinterpret_cast<float*>(u);
        if constexpr (MASK) {
          const int k0 = j * kBN;
#pragma unroll
          for (int c = 0; c < kBN; ++c) {
            const int key = k0 + c;
            if (key >= len_k_of<VARLEN>(T, p) || (CAUSAL && key > q_row + coff_of<VARLEN>(T, p))) s[c] = -INFINITY;
          }
        }
        // The exponentials are taken straight away against the running
        // reference maximum, and P goes into its buffer in two halves of 64
        // keys: the wait for P·V(g−1), the buffer's reader, sits between them,
        // by when it has long completed.  Only when a row has no reference
        // yet (its first visible block), or when its sum shows a key far
        // above the reference (Σp > 2^τ, so some p may exceed 2^τ; this also
        // catches an overflow to inf), does the warp compute the block
        // maximum, rescale where it moved by more than τ, and redo the
        // exponentials (S is still in registers).  The outputs are those of
        // computing the maximum first: a row that passes the sum test has no
        // key above m_run + τ, so it would not have been rescaled.
        // (Every row sees key 0 of its tile's first block, the only block where
        // m_run is still −inf.)
        bool redo = (j == 0);
        bool pv_seen = (g == 0);  // P·V(g−1) known complete (nothing before the CTA's first block)
        float lsum;
#pragma unroll 1
        for (;;) {
          if (redo) {
            float m8[8];  // row maximum (log2 domain): eight independent 16-wide chains
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
            const float mx =
                fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7])) * sc;
            const bool need = mx > m_run + p.tau;
            if (__any_sync(0xffffffffu, need)) {
              const float m_new = need ? mx : m_run;
              const float alpha = need ? ex2_mufu(m_run - m_new) : 1.f;
              if (j > 0) {
                // O holds the tile's blocks < j once the last P·V has landed.
                if (!rescale_o<L::D>(bar_pv_done, (g - 1) & 1, wc, tO, alpha)) return false;
                pv_seen = true;
              }
              l_run *= alpha;
              m_run = m_new;
              if constexpr (COUNT) {
                const unsigned int nres = __popc(__ballot_sync(0xffffffffu, need));
                if (lane == 0) atomicAdd(p.counters, static_cast<unsigned long long>(nres));
              }
            }
            __syncwarp();
          }
          // p = 2^(s·scale·log2 e − m_run), bf16 pairs, 64 keys at a time.
          const float negm = (m_run == -INFINITY) ? 0.f : -m_run;
          const uint64_t nm2 = pack2(negm, negm);
          uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float x0, x1;
              const int c = 64 * hh + 2 * i;
              unpack2(ffma2(pack2(s[c], s[c + 1]), sc2, nm2), x0, x1);
              if ((POLY >> (c / 16)) & 1u) {  // folded after unrolling
                ex2_poly2(x0, x1);
              } else {
                x0 = ex2_mufu(x0);
                x1 = ex2_mufu(x1);
              }
              acc[i & 3] = fadd2(acc[i & 3], pack2(x0, x1));
              pk[i] = pack_bf16x2(x0, x1);
            }
            if (hh == 0 && !pv_seen) {
              // The P buffer is free once P·V(g−1) has read it.
              const bool landed = wait_bar_cold(bar_pv_done, (g - 1) & 1, wc);
              if (__any_sync(0xffffffffu, !landed)) return false;
              tc_fence_after();
              pv_seen = true;
            }
            tmem_st32(tP + 32 * hh, pk);
          }
          float a0, a1, b0, b1;
          unpack2(fadd2(acc[0], acc[1]), a0, a1);
          unpack2(fadd2(acc[2], acc[3]), b0, b1);
          lsum = (a0 + a1) + (b0 + b1);
          if (redo || !__any_sync(0xffffffffu, !(lsum <= p.sum_limit))) break;
          redo = true;
        }
        // Test the next block's S without blocking; the answer is needed only
        // at that block's start, so the test's latency overlaps this block's end.
        s_ready = mbar_test_wait(bar_s_full, (g + 1) & 1);
        l_run += lsum;
        if constexpr (COUNT) {
          if (lane == 0) atomicAdd(p.counters + 1, 32ull);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar_p_full, lane);
        return true;
      };
      // Blocks whose keys all lie below Sk and, when causal, at or before the
      // tile's first row + coff need no mask.
      const int lk = len_k_of<VARLEN>(T, p);
      const int lim = CAUSAL ? min(lk, T.q0 + 1 + coff_of<VARLEN>(T, p)) : lk;
      const int n_full = min(T.nb, max(0, lim / kBN));
      int j = 0;
      for (; j < n_full && ok; ++j, ++g) ok = block(j, std::false_type{});
      for (; j < T.nb && ok; ++j, ++g) ok = block(j, std::true_type{});
      if (!ok) break;
      // ---------------------------------------------------- epilogue
      const bool landed = wait_bar(bar_o_final, tc & 1, wc);
      if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const int qb = tc & 1;
      uint8_t* const stage = smem + L::kQOff + qb * L::kTileBytes;
      // A packed sequence's last tile: each thread writes its own row (rows
      // beyond the sequence belong to the next one); else staged for the TMA
      // store.
      const bool direct = VARLEN && T.q0 + kBM > len_q_of<VARLEN>(T, p);
      uint16_t* const orow = o_row(T);
      uint32_t x[2][32];
      tmem_ld32(tO, x[0]);
      tmem_ld32(tO + 32, x[1]);
      tmem_wait_ld();
      reg_fence32(x[0]);
      reg_fence32(x[1]);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int q16 = 0; q16 < 4; ++q16) {  // four 16-byte chunks of 8 values
          uint4 wv;
          const uint32_t* o8 = &x[c][8 * q16];
          wv.x = pack_bf16x2(__uint_as_float(o8[0]) * inv, __uint_as_float(o8[1]) * inv);
          wv.y = pack_bf16x2(__uint_as_float(o8[2]) * inv, __uint_as_float(o8[3]) * inv);
          wv.z = pack_bf16x2(__uint_as_float(o8[4]) * inv, __uint_as_float(o8[5]) * inv);
          wv.w = pack_bf16x2(__uint_as_float(o8[6]) * inv, __uint_as_float(o8[7]) * inv);
          const int chunk = 4 * c + q16;  // 16-byte chunk of the 128-byte row
          if (!direct)
            *reinterpret_cast<uint4*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4)) = wv;
          else if (q_row < len_q_of<VARLEN>(T, p))
            *reinterpret_cast<uint4*>(orow + 8 * chunk) = wv;
        }
      }
      fence_proxy_async_smem();
      warp_arrive(bar_stage_full(qb), lane);  // the store warp writes the tile out
      if (q_row < len_q_of<VARLEN>(T, p)) {
        const float lse = (l_run > 0.f) ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        p.lse[lse0_of<VARLEN>(T, p) + r] = lse;
      }
      ++tc;
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

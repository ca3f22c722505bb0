// Exact attention forward kernel for sm_103a (GB300).
//
// One CTA computes two 128-row query tiles (Q0, Q1) of one (batch, head)
// against every visible 128-key block, with an online softmax, so the score
// matrix never leaves the chip ("FlashAttention 4: Atenção Mais Rápida …",
// section "Novidades no FlashAttention 4": tiles of Q, K, V streamed through
// on-chip memory, one CTA per output block set).
//
// Warp roles (320 threads):
//   warps 0-3  softmax group 0 — one thread per row of tile 0
//   warps 4-7  softmax group 1 — one thread per row of tile 1
//   warp  8    loader — TMA loads of Q0/Q1 once, then K_j, V_j into a ring of
//              shared-memory slots guarded by full/empty mbarriers
//   warp  9    MMA issuer (one thread) — tcgen05.mma S_t = Q_t K_jᵀ and
//              O_t += P_t V_j for both tiles in strict alternation,
//              accumulators in tensor memory (TMEM)
// This is the load → MMA → softmax → rescale → store pipeline of
// "FlashAttention 4: …", section "Novidades no FlashAttention 4" (warp
// specialisation), with the rescale step folded into the softmax warps: a row
// is rescaled only when its block maximum exceeds the running maximum by more
// than τ (section "Reescalonamento Softmax Online Mais Inteligente"), which
// after the first blocks is rare, so a separate correction warpgroup would
// mostly idle.  The two tiles ping-pong: while one softmax group works on its
// S tile, the tensor core runs the other tile's P·V and next Q·Kᵀ
// ("FlashAttention-3: …", section "Interleaving de GEMM e Softmax").
//
// TMEM columns (512 allocated): S0 [0,128), S1 [128,256), O0 [256, 256+D),
// O1 [256+D, 256+2D).  P_t (bf16, two per 32-bit column) overwrites the first
// 64 columns of S_t after the softmax thread has read its whole S row.
//
// Ordering rules the protocol relies on:
//  * tcgen05.mma operations issued by one thread execute in issue order, and
//    tcgen05.commit arrives only after all earlier ones complete.  The MMA
//    thread issues P_t(j−1)·V before S_t(j) = Q_t K_jᵀ, so S_t(j) never
//    overwrites P_t(j−1) early, and when s_full[t] fires for block j the O_t
//    update of block j−1 is finished — the softmax thread may rescale O_t.
//  * O_t is not touched by the MMA again until p_full[t] is signalled.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "attn_device.cuh"

namespace attn {

constexpr int kBM = 128;       // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;       // keys per block
constexpr int kThreads = 320;  // 8 softmax warps + loader + MMA issuer
constexpr int kLoaderWarp = 8;
constexpr int kMmaWarp = 9;    // MMA issuer; also allocates TMEM
constexpr uint32_t kTmemCols = 512;

struct FwdParams {
  float* lse;              // [B, H, Sq]
  unsigned int* status;    // device status word
  unsigned long long* counters;  // optional diagnostics (may be null)
  int B, H, Sq, Sk;
  int n_pairs;             // ceil(Sq / 256)
  float scale_log2;        // scale · log2(e)
  float tau;               // rescale threshold, log2 domain
  uint64_t timeout_ns;
  uint32_t test_flags;     // bit 0: loader withholds K/V (exercises the wait limit)
};

template <int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kSlabs = D / 64;                 // 128-byte-wide column slabs per row
  static constexpr uint32_t kSlabBytes = kBM * 128;     // one 128-row slab: 16 KB
  static constexpr uint32_t kTileBytes = kSlabBytes * kSlabs;
  static constexpr int kStages = (D == 128) ? 4 : 8;    // K/V ring slots (each holds one K or V tile)
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kRingOff = 2 * kTileBytes;
  static constexpr uint32_t kBarOff = kRingOff + kStages * kTileBytes;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], epi[2], done
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 2 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;  // tmem base (4 B) + abort flag (4 B)
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base to 1024
  __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(D) * t; }
};

__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]),
                 "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7]));
}

// POLY: bit c selects the FMA-pipe polynomial exp2 for 16-column chunk c of
// every 128-key block (compile time, so the exp loop is one basic block).
template <int D, bool CAUSAL, uint32_t POLY>
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
  const uint32_t bar_q = bars;
  auto bar_kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (1 + L::kStages + s); };
  auto bar_s_full = [&](int t) { return bars + 8u * (1 + 2 * L::kStages + t); };
  auto bar_p_full = [&](int t) { return bars + 8u * (3 + 2 * L::kStages + t); };
  auto bar_o_full = [&](int t) { return bars + 8u * (5 + 2 * L::kStages + t); };
  auto bar_epi = [&](int t) { return bars + 8u * (7 + 2 * L::kStages + t); };
  const uint32_t bar_done = bars + 8u * (9 + 2 * L::kStages);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (pair of query tiles, batch, head)
  const int BH = p.B * p.H;
  int pair, bh;
  if (CAUSAL) {  // heaviest query tiles first (longest-processing-time order)
    pair = p.n_pairs - 1 - static_cast<int>(blockIdx.x) / BH;
    bh = static_cast<int>(blockIdx.x) % BH;
  } else {  // the pairs of one head run side by side and share its K/V in L2
    pair = static_cast<int>(blockIdx.x) % p.n_pairs;
    bh = static_cast<int>(blockIdx.x) / p.n_pairs;
  }
  const int b = bh / p.H, h = bh % p.H;
  const int q0 = pair * 2 * kBM;
  const int ntiles = (p.Sq - q0 > kBM) ? 2 : 1;
  const int nk = (p.Sk + kBN - 1) / kBN;
  // Key blocks each tile visits (causal: up to the block holding its last row).
  const int nblk0 = CAUSAL ? min(nk, (min(q0 + kBM, p.Sq) - 1) / kBN + 1) : nk;
  const int nblk1 = CAUSAL ? min(nk, (min(q0 + 2 * kBM, p.Sq) - 1) / kBN + 1) : nk;
  auto nblk = [&](int t) { return t ? nblk1 : nblk0; };
  const int nmax = ntiles == 2 ? nblk1 : nblk0;

  // ---- set-up
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s_full(t), 1);
      mbar_init(bar_p_full(t), kBM);
      mbar_init(bar_o_full(t), 1);
      mbar_init(bar_epi(t), kBM);
    }
    mbar_init(bar_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == kLoaderWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (warp == kLoaderWarp) {
    // =========================================================== loader
    if (lane == 0) {
      int issued = 0;  // loads issued into the ring
      bool ok = true;
      mbar_arrive_expect_tx(bar_q, ntiles * L::kTileBytes);
      for (int t = 0; t < ntiles; ++t)
        for (int s = 0; s < L::kSlabs; ++s)
          tma_load_4d(sQ + t * L::kTileBytes + s * L::kSlabBytes, &tm_q, 64 * s, h, q0 + t * kBM, b, bar_q);
      if (p.test_flags & 1u) {
        // Test mode: no K/V copy is issued, so the MMA issuer's first wait
        // expires.  Only the Q copy is in flight; let it land and stop.
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_q, 0))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
      }
      for (int j = 0; j < nmax && ok && !(p.test_flags & 1u); ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = issued % L::kStages;
          const uint32_t ph = (issued / L::kStages) & 1u;
          if (!wait_bar(bar_kv_empty(slot), ph ^ 1u, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_kv_full(slot), L::kTileBytes);
          const CUtensorMap* m = kv ? &tm_v : &tm_k;
          for (int s = 0; s < L::kSlabs; ++s)
            tma_load_4d(sRing + slot * L::kTileBytes + s * L::kSlabBytes, m, 64 * s, h, j * kBN, b,
                        bar_kv_full(slot));
          ++issued;
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        const uint64_t t0 = globaltimer_ns();
        for (int n = (issued > L::kStages ? issued - L::kStages : 0); n < issued; ++n) {
          while (!mbar_try_wait(bar_kv_full(n % L::kStages), (n / L::kStages) & 1u))
            if (globaltimer_ns() - t0 > p.timeout_ns) break;
        }
        while (!mbar_try_wait(bar_q, 0))
          if (globaltimer_ns() - t0 > p.timeout_ns) break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ======================================================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false);
      constexpr uint32_t idPV = idesc_bf16(kBM, D, true);
      // Descriptor bases, computed once.  Every operand of the loop is a base
      // plus a constant (start address in 16-byte units; all shared-memory
      // offsets stay below 256 KB, so the 14-bit field never carries).
      const uint64_t dQ = sdesc_kmajor_sw128(sQ);
      const uint64_t dK = sdesc_kmajor_sw128(sRing);
      const uint64_t dV = sdesc_mnmajor_sw128(sRing, L::kSlabBytes);
      int consumed = 0;  // ring loads seen, in the loader's order K0, V0, K1, V1, …
      int v_prev_slot = 0;
      bool ok = wait_bar(bar_q, 0, wc);
      tc_fence_after();
      for (int j = 0; j <= nmax && ok; ++j) {
        int k_slot = -1;
        for (int t = 0; t < ntiles && ok; ++t) {
          const uint32_t tSt = tmem + L::col_s(t), tOt = tmem + L::col_o(t);
          if (j >= 1 && j <= nblk(t)) {
            // O_t (+)= P_t(j−1) · V_{j−1}
            if (!wait_bar(bar_p_full(t), (j - 1) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dv = dV + ((v_prev_slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts(tOt, tSt + kk * 8, dv + ((kk * 2048) >> 4), idPV, (j > 1 || kk > 0) ? 1u : 0u);
            if (j == nblk(t)) mma_commit(bar_o_full(t));
          }
          if (j < nblk(t)) {
            if (k_slot < 0) {
              k_slot = consumed % L::kStages;
              if (!wait_bar(bar_kv_full(k_slot), (consumed / L::kStages) & 1, wc)) { ok = false; break; }
              ++consumed;
              tc_fence_after();
            }
            // S_t = Q_t · K_jᵀ
            const uint64_t dq = dQ + ((t * L::kTileBytes) >> 4);
            const uint64_t dk = dK + ((k_slot * L::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk / 4) * L::kSlabBytes + (kk % 4) * 32) >> 4;
              mma_ss(tSt, dq + off, dk + off, idS, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar_s_full(t));
          }
        }
        if (!ok) break;
        if (j >= 1) mma_commit(bar_kv_empty(v_prev_slot));  // V_{j−1} no longer read
        if (j < nmax) {
          mma_commit(bar_kv_empty(k_slot));  // K_j no longer read
          const int vs = consumed % L::kStages;
          if (!wait_bar(bar_kv_full(vs), (consumed / L::kStages) & 1, wc)) { ok = false; break; }
          ++consumed;
          tc_fence_after();
          v_prev_slot = vs;
        }
      }
      // Every MMA issued above must finish before TMEM is released.
      mma_commit(bar_done);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_done, 0))
        if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
  } else {
    // ========================================================== softmax
    const int t = warp >> 2;              // tile handled by this warpgroup
    const int r = threadIdx.x & 127;      // row within the tile = TMEM lane
    if (t < ntiles) {
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + L::col_s(t) + lane_off;
      const uint32_t tO = tmem + L::col_o(t) + lane_off;
      const int q_tile = q0 + t * kBM;
      const int q_row = q_tile + r;
      const float sc = p.scale_log2;
      float m_run = -INFINITY;  // running reference maximum (log2 domain)
      float l_run = 0.f;        // running row sum (fp32, unrounded p)
      bool ok = true;
      const int nb = nblk(t);
      for (int j = 0; j < nb; ++j) {
        const bool got = wait_bar(bar_s_full(t), j & 1, wc);
        if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
        tc_fence_after();
        // Whole S row (128 fp32) in registers: four loads, one wait.
        uint32_t u[kBN];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&u[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32 * c]));
        float* const s = reinterpret_cast<float*>(u);
        const int k0 = j * kBN;
        if (k0 + kBN > p.Sk || (CAUSAL && k0 + kBN - 1 > q_tile)) {
#pragma unroll
          for (int c = 0; c < kBN; ++c) {
            const int key = k0 + c;
            if (key >= p.Sk || (CAUSAL && key > q_row)) s[c] = -INFINITY;
          }
        }
        // Row maximum as a tree of eight independent 16-wide chains.
        float m8[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float* x = s + 16 * g;
          float a = fmax3(x[0], x[1], x[2]);
          float b2 = fmax3(x[3], x[4], x[5]);
          a = fmax3(a, x[6], x[7]);
          b2 = fmax3(b2, x[8], x[9]);
          a = fmax3(a, x[10], x[11]);
          b2 = fmax3(b2, x[12], x[13]);
          m8[g] = fmax3(a, b2, fmaxf(x[14], x[15]));
        }
        float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        mx *= sc;
        const bool need = mx > m_run + p.tau;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mx : m_run;
          const float alpha = need ? ex2_mufu(m_run - m_new) : 1.f;
          if (j > 0) {  // O_t holds blocks < j: scale it (block j−1's P·V has completed)
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + 32 * c, o);
              tmem_wait_ld();
              reg_fence32(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + 32 * c, o);
            }
          }
          l_run *= alpha;
          m_run = m_new;
          if (p.counters != nullptr) {
            const unsigned int nres = __popc(__ballot_sync(0xffffffffu, need));
            if (lane == 0) atomicAdd(p.counters, static_cast<unsigned long long>(nres));
          }
        }
        if (p.counters != nullptr && lane == 0) atomicAdd(p.counters + 1, 32ull);
        __syncwarp();
        const float negm = (m_run == -INFINITY) ? 0.f : -m_run;
        const uint64_t sc2 = pack2(sc, sc);
        const uint64_t nm2 = pack2(negm, negm);
        uint64_t acc[4] = {0, 0, 0, 0};  // four packed partial sums (+0.0f pairs)
#pragma unroll
        for (int ch = 0; ch < kBN / 16; ++ch) {
          uint32_t pk[8];
          constexpr uint32_t kPoly = POLY;
          const bool use_poly = (kPoly >> ch) & 1u;  // folded after unrolling
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
            pk[i] = pack_bf16x2(x0, x1);
          }
          tmem_st8(tS + ch * 8, pk);
        }
        float a0, a1, b0, b1;
        unpack2(fadd2(acc[0], acc[1]), a0, a1);
        unpack2(fadd2(acc[2], acc[3]), b0, b1);
        l_run += (a0 + a1) + (b0 + b1);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_p_full(t));
      }
      // ------------------------------------------------------ epilogue
      if (ok) {
        const bool got = wait_bar(bar_o_full(t), 0, wc);
        ok = !__any_sync(0xffffffffu, !got);
      }
      if (ok) {
        tc_fence_after();
        const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
        // Stage O_t in its (now idle) Q_t buffer with the 128-byte swizzle
        // the TMA store expects: 16-byte chunk c of row r sits at c ^ (r % 8).
        uint8_t* const stage = smem + L::kQOff + t * L::kTileBytes;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
          reg_fence32(o);
          const int slab = c / 2;
#pragma unroll
          for (int q16 = 0; q16 < 4; ++q16) {  // four 16-byte chunks of 8 values
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * q16 + 0]) * inv_l, __uint_as_float(o[8 * q16 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[8 * q16 + 2]) * inv_l, __uint_as_float(o[8 * q16 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[8 * q16 + 4]) * inv_l, __uint_as_float(o[8 * q16 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[8 * q16 + 6]) * inv_l, __uint_as_float(o[8 * q16 + 7]) * inv_l);
            const int chunk = (c % 2) * 4 + q16;
            *reinterpret_cast<uint4*>(stage + slab * L::kSlabBytes + r * 128 + ((chunk ^ (r & 7)) * 16)) = w;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_epi(t));
        if (q_row < p.Sq) {
          const float lse = (l_run > 0.f) ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
          p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + q_row] = lse;
        }
        if (r == 0) {
          if (wait_bar(bar_epi(t), 0, wc)) {
            const uint32_t src = smem_u32(stage);
            for (int s = 0; s < L::kSlabs; ++s)
              tma_store_4d(&tm_o, src + s * L::kSlabBytes, 64 * s, h, q_tile, b);
            tma_store_commit();
            tma_store_wait_read0();  // smem may be released; the global writes complete on their own
          }
        }
      }
    }
  }

  // ---- tear-down: every role arrives here; all TMEM reads/writes are done
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn

// bwd_dual_tc.cuh -- tensor-core kernels (tcgen05 + TMEM + TMA) for the
// reverse mode of the dual computation, fp16/bf16 inputs, fp32 accumulation.
//
// With P = exp(S - lse) recomputed from the saved log-sum-exp, the backward
// needs no online softmax: every (row, key) term is independent once the
// per-row scalars lse, mu, nu = gtO.O and delta = gO.O + gtO.tO - mu*nu are
// known.  Per (b, h):
//   dS  = s (dQ K^T + Q dK^T)     G = gtO V^T     gP1 = gO V^T + gtO dV^T
//   gP  = gP1 + G (dS - mu) - nu dS
//   gS  = P (gP - delta)          g_dS = P (G - nu)          dP = P (dS - mu)
//   gQ  = s (gS K + g_dS dK)      g_dQ = s g_dS K
//   gK  = s (gS^T Q + g_dS^T dQ)  g_dK = s g_dS^T Q
//   gV  = P^T gO + dP^T gtO       g_dV = P^T gtO
//
// Query-major kernel (gQ, g_dQ): one CTA per 128-row query tile, looping over
// 64-key tiles; like the forward, the score products take their A operands
// (Q, dQ, gO, gtO) from shared memory:
//   [S | Q dK^T]      = Q   [K ; dK]^T      then  Q dK^T += dQ K^T
//   [G | gtO dV^T]    = gtO [V ; dV]^T      then  gtO dV^T += gO V^T   (= gP1)
// the elementwise warps turn each 64-key tile into gS and g_dS (16-bit, in
// TMEM over the S columns they read), and
//   [g_dQ | gQ] += g_dS [K | dK]            then  gQ += gS K
// with the same shared-memory K/dK tile read as an MN-major operand.
//
// Key-major kernel (gK, g_dK, gV, g_dV): one CTA per 128-key tile, looping over
// query tiles (64 rows for the value part, 32 when the four score matrices
// of the key part share a TMEM buffer), with the transposed scores (TMEM
// lanes = keys):
//   [S^T | K dQ^T]    = K [Q ; dQ]^T        then  K dQ^T += dK Q^T
//   [G^T | V gO^T]    = V [gtO ; gO]^T      then  V gO^T += dV gtO^T   (= gP1^T)
//   [g_dV | gV] += P^T [gtO | gO],  gV += dP^T gtO
//   [g_dK | gK] += g_dS^T [Q | dQ], gK += gS^T Q
// At D = 128 the four key-side accumulators do not fit TMEM next to the
// scores, so the key-major kernel runs twice (value part, key part).
//
// Each kernel: warp 0 TMA producer, warp 1 TMEM allocator and issuer of the
// first group of score products, warps 2..9 two elementwise warpgroups (each
// owns half of the columns of a tile, a thread owns a TMEM lane).  The second
// group of score products ([G | gP], disjoint TMEM columns) has its own
// issuing warp (query-major: warp 10; key-major key part: warp 11), and the
// key-major kernel's accumulate products another (warp 10).  The query-major
// kernel's accumulate products are issued by warp 1 too: after the score
// products of the same tile when [S | dS] has one TMEM buffer (D = 128), or
// with two buffers (D = 64, and the primal) after the next tile's score
// products, so those run while the elementwise warps work.  After the row
// pass the query-major and key-major kernels are independent; the host puts
// the key-major ones on a second stream.  Every wait is bounded.
//
// The PRIMAL specialisation is the backward of attention without tangents
// (dQ = dK = dV = 0, gtO = 0): only S, gP1 = gO V^T, gS and the gQ, gK, gV
// products remain (see the kernels below).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "fwd_dual_tc.cuh"

namespace jvp {

// Query-major kernel: warp 0 TMA, warp 1 the [S | dS] score products and the
// accumulate MMAs, warps 2..9 elementwise, warp 10 the [G | gP] score products.
constexpr int kBwdThreads = 96 + 256;
constexpr int kBwdScoreWarpQ = 10;
// The key-major kernel adds a warp (10) that issues the accumulate MMAs while
// warp 1 issues the score products, and (key part) a warp (11) that issues
// the second, independent group of score products.
constexpr int kBwdThreadsK = 128 + 256;
constexpr int kBwdAccWarp = 10;
constexpr int kBwdScoreWarpB = 11;

// ----------------------------------------------------------------------------
// Query-major kernel.
template <int D, bool PRIMAL = false>
struct BqLayout {
  static constexpr int BM = 128;  // query rows per CTA
  static constexpr int BN = 64;   // keys per tile
  static constexpr int KCH = D / 64;
  // [K ; dK] stays until the accumulate MMAs, [V ; dV] is freed after the
  // score MMAs: at D = 128 two K stages and one V stage fit next to the 128 KB
  // of resident query-side tiles, so the next K tile loads during the current
  // tile's elementwise stage and accumulate MMAs.
  // The primal keeps only Q and gO resident (the dQ and gtO slots go to a
  // third K stage and a second V stage at D = 128).
  static constexpr int NSK = (D == 64 || PRIMAL) ? 3 : 2;
  static constexpr int NSV = (D == 64) ? 3 : PRIMAL ? 2 : 1;
  static constexpr int QT_BYTES = KCH * BM * 128;  // one [128 x D] query-side tile
  static constexpr int KCHUNK = 2 * BN * 128;      // [K rows | dK rows] of one 64-column chunk
  static constexpr int KBLK = KCH * KCHUNK;        // [K ; dK] block of one stage
  static constexpr int OFF_Q = 0, OFF_DQ = QT_BYTES;  // (dQ, gtO: not in the primal)
  static constexpr int OFF_GO = (PRIMAL ? 1 : 2) * QT_BYTES, OFF_GTO = 3 * QT_BYTES;
  static constexpr int OFF_K = (PRIMAL ? 2 : 4) * QT_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * KBLK;
  static constexpr int OFF_CTRL = OFF_V + NSV * KBLK;
  static constexpr int CTRL_BYTES = 512;
  static constexpr int SMEM_BYTES = OFF_CTRL + CTRL_BYTES + 1024;
  // TMEM columns: NBS buffers of [S | dS] (128 columns each), then [G | gP],
  // then the accumulators.  Two buffers where the accumulators leave room
  // (D = 64: [g_dQ | gQ] is 128 columns; the primal has gQ alone), so tile
  // t+1's [S | dS] products run while the elementwise warps work on tile t.
  static constexpr int NBS = (D == 64 || PRIMAL) ? 2 : 1;
  static constexpr uint32_t TM_S = 0, TM_DS = 64;  // + 128 * buffer
  static constexpr uint32_t TM_G = NBS * 128, TM_GP = TM_G + 64, TM_ACC = TM_G + 128;
  static constexpr uint32_t A_GQ = PRIMAL ? 0 : D;  // gQ within the accumulators
  static_assert(TM_ACC + A_GQ + D <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

template <int NSK, int NSV>
struct BwdCtrl {
  uint64_t q_full;
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  uint64_t s_full[2];  // [S | dS] of a buffer (warp 1)
  uint64_t g_full[2];  // [G | gP] (warp 10; the primal's gP of each buffer has its own)
  uint64_t p_full[2];  // the elementwise warps are done with a buffer's tile
  uint64_t o_full, drain, drain_b;
  uint32_t tmem_base;
  int abort;
};

// Per-(row, key) backward terms from the score-side values; xm is the
// base-2 logit minus the row's base-2 log-sum-exp.  keep = false gives
// all-zero terms (masked key, or a row that keeps no key).
// One key's mask entries for N query rows (key-major kernel): loaded one by
// one (the rows are strided in memory), all before they are needed.
template <int MASK, int N>
struct MaskCol {  // no per-entry data for none / causal
  __device__ __forceinline__ void load(int, const void*, long long) {}
  __device__ __forceinline__ bool keep(int) const { return true; }
  __device__ __forceinline__ float add(int) const { return 0.f; }
};
template <int N>
struct MaskCol<kMaskBool, N> {
  uint32_t v[N];
  __device__ __forceinline__ void load(int r, const void* m, long long idx) {
    v[r] = static_cast<const uint8_t*>(m)[idx];
  }
  __device__ __forceinline__ bool keep(int r) const { return v[r] != 0u; }
  __device__ __forceinline__ float add(int) const { return 0.f; }
};
template <int N>
struct MaskCol<kMaskAdditive, N> {
  float v[N];
  __device__ __forceinline__ void load(int r, const void* m, long long idx) {
    v[r] = static_cast<const float*>(m)[idx];
  }
  __device__ __forceinline__ bool keep(int) const { return true; }
  __device__ __forceinline__ float add(int r) const { return v[r]; }
};

struct BwdTerms {
  float gS, gdS, P, dP;
};
__device__ __forceinline__ BwdTerms bwd_terms(bool keep, float xm, float ds_raw, float g,
                                              float gp1, float s, float mu, float nu,
                                              float delta) {
  BwdTerms r;
  const float P = keep ? ex2_approx(xm) : 0.0f;
  const float dS = s * ds_raw;
  const float gP = fmaf(g, dS - mu, gp1) - nu * dS;
  r.P = P;
  r.dP = P * (dS - mu);
  r.gS = P * (gP - delta);
  r.gdS = P * (g - nu);
  return r;
}

// PRIMAL: the backward of attention without tangents (dQ = dK = dV = 0 and
// gtO = 0, so dS, G, g_dS and the tangent gradients vanish): only S = Q K^T
// and gP1 = gO V^T are formed, gS = P (gP1 - delta), and gQ += gS K.  The
// tangent operands are neither loaded nor multiplied.
template <typename T, int D, int MASK, bool PRIMAL = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_q_tc_kernel(const __grid_constant__ BwdTcMaps maps, const BwdParams p, int group_heads,
                    unsigned int* status) {
  using L = BqLayout<D, PRIMAL>;
  constexpr int NSK = L::NSK, NSV = L::NSV, BN = L::BN, BM = L::BM;
  constexpr int NBS = L::NBS;
  constexpr bool kBF16 = ElemTraits<T>::kBF16;
  constexpr int KSD = D / 16;   // K-steps over the head dimension
  constexpr int KSN = BN / 16;  // K-steps over a key tile
  constexpr uint32_t I_N128 = idesc_f16(kBF16, 128, 128, false);
  constexpr uint32_t I_N64 = idesc_f16(kBF16, 128, 64, false);
  constexpr uint32_t I_ACC2 = idesc_f16(kBF16, 128, 2 * D, true);  // D = 64: [g_dQ | gQ]
  constexpr uint32_t I_ACC1 = idesc_f16(kBF16, 128, D, true);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  static_assert(sizeof(BwdCtrl<NSK, NSV>) <= L::CTRL_BYTES, "control block budget");
  BwdCtrl<NSK, NSV>* ctrl = reinterpret_cast<BwdCtrl<NSK, NSV>*>(smem + L::OFF_CTRL);
  volatile int* abort = &ctrl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int BH = p.B * p.H;
  const int nq = (p.Nq + BM - 1) / BM;
  const int G = group_heads;
  // Query-major split: the qsplits CTAs of one query tile are adjacent.
  const int QS = p.qsplits > 1 ? p.qsplits : 1;
  const int split = static_cast<int>(blockIdx.x % QS);
  const int item = static_cast<int>(blockIdx.x / QS);
  const int g = item / (G * nq);
  const int rem = item - g * G * nq;
  const int Gg = min(G, BH - g * G);
  const int q_rank = rem / Gg;
  const int bh = g * G + rem % Gg;
  // Causal alone, or on top of a bool / additive mask (runtime flag).
  const bool causal =
      (MASK == kMaskCausal) || ((MASK == kMaskBool || MASK == kMaskAdditive) && p.causal != 0);
  const int qt = causal ? nq - 1 - q_rank : q_rank;
  const int b = bh / p.H, h = bh % p.H;
  const int hk = h / p.kv_group;  // key/value head (grouped-query attention)
  const int q0 = qt * BM;
  int n_all = (p.Nk + BN - 1) / BN;
  if (causal) n_all = min(n_all, (min(q0 + BM, p.Nq) - 1) / BN + 1);
  // This CTA's key tiles [kv_lo, kv_lo + n_kv) (all of them unless split).
  const int per_split = (n_all + QS - 1) / QS;
  const int kv_lo = min(n_all, split * per_split);
  const int n_kv = min(n_all, kv_lo + per_split) - kv_lo;

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&ctrl->k_full[s], 1);
      mbar_init(&ctrl->k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&ctrl->v_full[s], 1);
      mbar_init(&ctrl->v_empty[s], 1);
    }
    // With one [S | dS] buffer both score groups complete s_full[0] (two
    // commits); with two, [G | gP] has its own barrier (warp 1 may commit the
    // next buffer's products before warp 10 commits this tile's).
    for (int u = 0; u < 2; ++u) {
      mbar_init(&ctrl->s_full[u], (NBS == 1 && u == 0) ? 2 : 1);
      mbar_init(&ctrl->p_full[u], 256);
    }
    mbar_init(&ctrl->g_full[0], 1);
    mbar_init(&ctrl->g_full[1], 1);
    mbar_init(&ctrl->o_full, 1);
    mbar_init(&ctrl->drain, 1);
    mbar_init(&ctrl->drain_b, 1);
    ctrl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctrl->q_full, (PRIMAL ? 2 : 4) * L::QT_BYTES);
      for (int c = 0; c < L::KCH; ++c) {
        const int o = c * BM * 128;
        tma_load_4d(smem + L::OFF_Q + o, &maps.q, &ctrl->q_full, c * 64, q0, h, b);
        tma_load_4d(smem + L::OFF_GO + o, &maps.go, &ctrl->q_full, c * 64, q0, h, b);
        if (!PRIMAL) {
          tma_load_4d(smem + L::OFF_DQ + o, &maps.dq, &ctrl->q_full, c * 64, q0, h, b);
          tma_load_4d(smem + L::OFF_GTO + o, &maps.gto, &ctrl->q_full, c * 64, q0, h, b);
        }
      }
      int kf = 0, vf = 0;
      for (int t = 0; t < n_kv; ++t) {
        const int sk = t % NSK, sv = t % NSV;
        const int j0 = (kv_lo + t) * BN;
        if (!mbar_wait(&ctrl->k_empty[sk], ((t / NSK) & 1) ^ 1, abort)) {
          record_timeout(status, abort);
          break;
        }
        uint8_t* kb = smem + L::OFF_K + sk * L::KBLK;
        mbar_arrive_expect_tx(&ctrl->k_full[sk], PRIMAL ? L::KBLK / 2 : L::KBLK);
        for (int c = 0; c < L::KCH; ++c) {
          tma_load_4d(kb + c * L::KCHUNK, &maps.k, &ctrl->k_full[sk], c * 64, j0, hk, b);
          if (!PRIMAL)
            tma_load_4d(kb + c * L::KCHUNK + BN * 128, &maps.dk, &ctrl->k_full[sk], c * 64, j0, hk,
                        b);
        }
        ++kf;
        if (!mbar_wait(&ctrl->v_empty[sv], ((t / NSV) & 1) ^ 1, abort)) {
          record_timeout(status, abort);
          break;
        }
        uint8_t* vb = smem + L::OFF_V + sv * L::KBLK;
        mbar_arrive_expect_tx(&ctrl->v_full[sv], PRIMAL ? L::KBLK / 2 : L::KBLK);
        for (int c = 0; c < L::KCH; ++c) {
          tma_load_4d(vb + c * L::KCHUNK, &maps.v, &ctrl->v_full[sv], c * 64, j0, hk, b);
          if (!PRIMAL)
            tma_load_4d(vb + c * L::KCHUNK + BN * 128, &maps.dv, &ctrl->v_full[sv], c * 64, j0, hk,
                        b);
        }
        ++vf;
      }
      if (*abort) {
        const int zero = 0;
        mbar_wait(&ctrl->q_full, 0, &zero);
        for (int t = max(0, kf - NSK); t < kf; ++t)
          mbar_wait(&ctrl->k_full[t % NSK], (t / NSK) & 1, &zero);
        for (int t = max(0, vf - NSV); t < vf; ++t)
          mbar_wait(&ctrl->v_full[t % NSV], (t / NSV) & 1, &zero);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(&ctrl->q_full, 0, abort);
      tc_fence_after();
      const uint32_t aQ = smem_u32(smem + L::OFF_Q), adQ = smem_u32(smem + L::OFF_DQ);
      // [S | dS] of tile t goes into buffer t % NBS.  With two buffers the
      // products of tile t are issued before the accumulate MMAs of tile
      // t - 1 (which read gS, g_dS from the other buffer), so they run while
      // the elementwise warps work on tile t - 1; with one buffer they follow
      // them in issue order.  Warp 10 fills [G | gP] meanwhile.
      auto issue_scores = [&](int t) -> bool {
        const int sk = t % NSK;
        if (!mbar_wait(&ctrl->k_full[sk], (t / NSK) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + L::OFF_K + sk * L::KBLK);
        const uint32_t sb = tmem + (t % NBS) * 128;
#pragma unroll
        for (int kk = 0; kk < KSD; ++kk) {  // [S | Q dK^T] = Q [K ; dK]^T  (primal: S = Q K^T)
          const uint32_t off = (kk & 3) * 32;
          mma_ss(sb + L::TM_S, sdesc_sw128(aQ + (kk >> 2) * BM * 128 + off, 16, 1024),
                 sdesc_sw128(kb + (kk >> 2) * L::KCHUNK + off, 16, 1024),
                 PRIMAL ? I_N64 : I_N128, kk > 0);
        }
        if (!PRIMAL) {
#pragma unroll
          for (int kk = 0; kk < KSD; ++kk) {  // Q dK^T += dQ K^T
            const uint32_t off = (kk & 3) * 32;
            mma_ss(sb + L::TM_DS, sdesc_sw128(adQ + (kk >> 2) * BM * 128 + off, 16, 1024),
                   sdesc_sw128(kb + (kk >> 2) * L::KCHUNK + off, 16, 1024), I_N64, 1u);
          }
        }
        mma_commit(&ctrl->s_full[t % NBS]);
        return true;
      };
      auto issue_accumulate = [&](int t) -> bool {
        if (!mbar_wait(&ctrl->p_full[t & 1], (t >> 1) & 1, abort)) return false;
        tc_fence_after();
        const int sk = t % NSK;
        const uint32_t kb = smem_u32(smem + L::OFF_K + sk * L::KBLK);
        const uint32_t sb = tmem + (t % NBS) * 128;
        // gS and g_dS of keys [16 kk, 16 kk + 16) (warpgroup kk / 2, half
        // kk % 2): gS at columns 16 kk, g_dS at 16 kk + 8 of the buffer.
#pragma unroll
        for (int kk = 0; kk < KSN && !PRIMAL; ++kk) {
          const uint32_t a_gs = sb + kk * 16;
          const uint32_t a_gds = a_gs + 8;
          const uint32_t kx = kb + kk * 16 * 128;  // MN-major: 16 keys per K-step
          const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
          if (D == 64) {
            // [g_dQ | gQ] += g_dS [K | dK]  (K and dK chunks 8 KB apart)
            mma_ts(tmem + L::TM_ACC, a_gds, sdesc_sw128(kx, BN * 128, 1024), I_ACC2, acc);
          } else {
            // g_dQ += g_dS K ; gQ += g_dS dK  (chunks of one tensor 16 KB apart)
            mma_ts(tmem + L::TM_ACC, a_gds, sdesc_sw128(kx, L::KCHUNK, 1024), I_ACC1, acc);
            mma_ts(tmem + L::TM_ACC + D, a_gds, sdesc_sw128(kx + BN * 128, L::KCHUNK, 1024),
                   I_ACC1, acc);
          }
        }
#pragma unroll
        for (int kk = 0; kk < KSN; ++kk) {  // gQ += gS K  (the first products of the primal)
          const uint32_t a_gs = sb + kk * 16;
          mma_ts(tmem + L::TM_ACC + L::A_GQ, a_gs,
                 sdesc_sw128(kb + kk * 16 * 128, D == 64 ? BN * 128 : L::KCHUNK, 1024), I_ACC1,
                 PRIMAL ? ((t > 0 || kk > 0) ? 1u : 0u) : 1u);
        }
        mma_commit(&ctrl->k_empty[sk]);
        return true;
      };
      for (int t = 0; ok && t <= n_kv; ++t) {
        if (NBS == 2) {
          if (t < n_kv && !issue_scores(t)) ok = false;
          if (ok && t > 0 && !issue_accumulate(t - 1)) ok = false;
        } else {
          if (t > 0 && !issue_accumulate(t - 1)) ok = false;
          if (ok && t < n_kv && !issue_scores(t)) ok = false;
        }
      }
      if (ok) mma_commit(&ctrl->o_full);
      if (!ok) record_timeout(status, abort);
      mma_commit(&ctrl->drain);
      const int zero = 0;
      mbar_wait(&ctrl->drain, 0, &zero);
    }
  } else if (warp == kBwdScoreWarpQ) {
    // ------------------------------------------------------------ [G | gP] score MMAs
    // [G | gP] (one buffer) is free for tile t once the elementwise warps are
    // done with tile t - 1 (the accumulate MMAs read only the [S | dS] buffers).
    if (lane == 0) {
      bool ok = mbar_wait(&ctrl->q_full, 0, abort);
      tc_fence_after();
      const uint32_t aGO = smem_u32(smem + L::OFF_GO), aGTO = smem_u32(smem + L::OFF_GTO);
      // The primal's gP of tile t goes into the free half of score buffer
      // t % 2 (no dS there), so it waits only for the elementwise warps to be
      // done with tile t - 2, the buffer's previous tile.
      constexpr int kLag = PRIMAL ? 2 : 1;
      for (int t = 0; ok && t < n_kv; ++t) {
        const int sv = t % NSV;
        if ((t >= kLag &&
             !mbar_wait(&ctrl->p_full[(t - kLag) & 1], ((t - kLag) >> 1) & 1, abort)) ||
            !mbar_wait(&ctrl->v_full[sv], (t / NSV) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vb = smem_u32(smem + L::OFF_V + sv * L::KBLK);
        if (!PRIMAL) {
#pragma unroll
          for (int kk = 0; kk < KSD; ++kk) {  // [G | gtO dV^T] = gtO [V ; dV]^T
            const uint32_t off = (kk & 3) * 32;
            mma_ss(tmem + L::TM_G, sdesc_sw128(aGTO + (kk >> 2) * BM * 128 + off, 16, 1024),
                   sdesc_sw128(vb + (kk >> 2) * L::KCHUNK + off, 16, 1024), I_N128, kk > 0);
          }
        }
#pragma unroll
        for (int kk = 0; kk < KSD; ++kk) {  // gtO dV^T += gO V^T  (primal: gP1 = gO V^T)
          const uint32_t off = (kk & 3) * 32;
          mma_ss(tmem + (PRIMAL ? (t % NBS) * 128 + L::TM_DS : L::TM_GP),
                 sdesc_sw128(aGO + (kk >> 2) * BM * 128 + off, 16, 1024),
                 sdesc_sw128(vb + (kk >> 2) * L::KCHUNK + off, 16, 1024), I_N64,
                 PRIMAL ? (kk > 0 ? 1u : 0u) : 1u);
        }
        mma_commit(&ctrl->v_empty[sv]);
        mma_commit(NBS == 1 ? &ctrl->s_full[0] : &ctrl->g_full[PRIMAL ? (t & 1) : 0]);
      }
      if (!ok) record_timeout(status, abort);
      mma_commit(&ctrl->drain_b);
      const int zero = 0;
      mbar_wait(&ctrl->drain_b, 0, &zero);
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ elementwise
    const int wg = (warp - 2) >> 2;
    const int sub = warp & 3;
    const int r = sub * 32 + lane;
    const int i = q0 + r;
    const bool row_ok = i < p.Nq;
    const uint32_t lb = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const long long ridx = static_cast<long long>(bh) * p.Nq + (row_ok ? i : 0);
    const bool rd = row_ok && JVP_CHECK(ridx < static_cast<long long>(p.B) * p.H * p.Nq, status,
                                        kChkGlobalRow);
    const float lse = rd ? p.lse[ridx] : -INFINITY;
    const float lse2 = lse * kLog2e;
    const bool live = rd && lse != -INFINITY;
    const float mu = (rd && !PRIMAL) ? p.mu[ridx] : 0.f;
    const float nu = (rd && !PRIMAL) ? p.nu[ridx] : 0.f;
    const float delta = rd ? p.delta[ridx] : 0.f;
    const float c = p.scale * kLog2e;
    const float s = p.scale;
    bool ok = true;
    const void* mrow = nullptr;
    if (MASK == kMaskBool || MASK == kMaskAdditive) {
      const long long off = static_cast<long long>(b) * p.msb + static_cast<long long>(h) * p.msh +
                            static_cast<long long>(row_ok ? i : 0) * p.msq;
      mrow = (MASK == kMaskBool)
                 ? static_cast<const void*>(static_cast<const uint8_t*>(p.mask) + off)
                 : static_cast<const void*>(static_cast<const float*>(p.mask) + off);
    }
    // The row-scalar loads above are plain global reads of the workspace and
    // outputs of earlier kernels on this stream.
    FwdParams mp{};  // only the mask fields are used by MaskRegs
    mp.Nk = p.Nk;
    mp.msk = p.msk;
    mp.mask_vec = p.mask_vec;
    // One half of this warpgroup's 32 keys of a tile: gS and g_dS go into
    // the 16 columns of S the half has just read (gS first, g_dS next), so
    // the other half's inputs stay intact.
    // sb: the [S | dS] buffer's first column.
    auto half = [&](int j0h, uint32_t sb, uint32_t col, const MaskRegs<MASK, 16>& mreg) {
      uint32_t rs[16], rds[16], rg[16], rgp[16];
      const bool cols_ok = JVP_CHECK(L::TM_GP + col + 16 <= 512u &&
                                         sb + L::TM_DS + col + 16 <= L::TM_G,
                                     status, kChkTmem);
      if (PRIMAL) {
#pragma unroll
        for (int e = 0; e < 16; ++e) rds[e] = rg[e] = 0u;  // dS = G = 0
        if (cols_ok) tmem_ld16x2(lb + sb + L::TM_S + col, lb + sb + L::TM_DS + col, rs, rgp);
      } else if (cols_ok) {
        tmem_ld16x2(lb + sb + L::TM_S + col, lb + sb + L::TM_DS + col, rs, rds);
        tmem_ld16x2(lb + L::TM_G + col, lb + L::TM_GP + col, rg, rgp);
      }
      uint32_t pgs[8], pgds[8];
#pragma unroll
      for (int jj = 0; jj < 16; jj += 2) {
        float gs[2], gds[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0h + jj + e;
          bool keep = live && j < p.Nk;
          float x = fmaf(__uint_as_float(rs[jj + e]), c, -lse2);
          if (causal) keep = keep && j <= i;
          if constexpr (MASK == kMaskBool) keep = keep && mreg.keep(jj + e);
          if constexpr (MASK == kMaskAdditive) {
            x = fmaf(mreg.a[jj + e], kLog2e, x);
            keep = keep && x != -INFINITY;
          }
          const BwdTerms bt =
              bwd_terms(keep, x, __uint_as_float(rds[jj + e]), __uint_as_float(rg[jj + e]),
                        __uint_as_float(rgp[jj + e]), s, mu, nu, delta);
          gs[e] = bt.gS;
          gds[e] = bt.gdS;
        }
        pgs[jj >> 1] = ElemTraits<T>::pack(gs[0], gs[1]);
        pgds[jj >> 1] = ElemTraits<T>::pack(gds[0], gds[1]);
      }
      if (cols_ok) {
        tmem_st8(lb + sb + col, pgs);
        if (!PRIMAL) tmem_st8(lb + sb + col + 8, pgds);
      }
    };
    // The mask entries of this warpgroup's 32 keys of a tile are loaded one
    // tile ahead, so their latency overlaps a whole tile of work.
    MaskRegs<MASK, 16> n0, n1;
    if (row_ok && n_kv > 0) {
      n0.load(mp, mrow, kv_lo * BN + wg * 32);
      n1.load(mp, mrow, kv_lo * BN + wg * 32 + 16);
    }
    for (int t = 0; t < n_kv; ++t) {
      const int j0 = (kv_lo + t) * BN + wg * 32;
      const MaskRegs<MASK, 16> m0 = n0, m1 = n1;
      if (row_ok && t + 1 < n_kv) {
        n0.load(mp, mrow, j0 + BN);
        n1.load(mp, mrow, j0 + BN + 16);
      }
      if (!warp_wait(&ctrl->s_full[t % NBS], (t / NBS) & 1, status, abort) ||
          (NBS == 2 && !warp_wait(&ctrl->g_full[PRIMAL ? (t & 1) : 0],
                                  PRIMAL ? ((t >> 1) & 1) : (t & 1), status, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sb = static_cast<uint32_t>(t % NBS) * 128;
      half(j0, sb, wg * 32, m0);
      half(j0 + 16, sb, wg * 32 + 16, m1);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctrl->p_full[t & 1]);
    }
    if (ok && n_kv > 0) ok = warp_wait(&ctrl->o_full, 0, status, abort);
    if (ok && !(PRIMAL && wg == 0)) {
      tc_fence_after();
      // Warpgroup 0 writes g_dQ, warpgroup 1 writes gQ (both scaled by s);
      // the primal has gQ alone.
      void* dst = wg == 0 ? p.g_dq : p.g_q;
      const uint32_t acol = L::TM_ACC + (wg == 0 ? 0u : L::A_GQ);
      const Strides& ds = wg == 0 ? p.sgdq : p.sgq;
      T* row = static_cast<T*>(dst) + static_cast<long long>(b) * ds.b +
               static_cast<long long>(h) * ds.h + static_cast<long long>(row_ok ? i : 0) * ds.n;
      // split: this CTA's fp32 partial row (slot 0 g_dQ, 1 gQ)
      float* prow = p.qws + ((static_cast<long long>(split) * 2 + wg) * BH + bh) *
                                static_cast<long long>(p.Nq) * D +
                    static_cast<long long>(row_ok ? i : 0) * D;
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        uint32_t a[32];
        if (n_kv > 0 && JVP_CHECK(acol + col + 32 <= 512u, status, kChkTmem)) {
          tmem_ld32(lb + acol + col, a);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = 0u;
        }
        if (QS > 1) {
          if (row_ok && JVP_CHECK(i < p.Nq, status, kChkGlobalCol)) {
            float4* pd = reinterpret_cast<float4*>(prow + col);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              pd[v4] = make_float4(__uint_as_float(a[4 * v4]) * s, __uint_as_float(a[4 * v4 + 1]) * s,
                                   __uint_as_float(a[4 * v4 + 2]) * s,
                                   __uint_as_float(a[4 * v4 + 3]) * s);
          }
          continue;
        }
        uint32_t po[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          po[e >> 1] = ElemTraits<T>::pack(__uint_as_float(a[e]) * s, __uint_as_float(a[e + 1]) * s);
        if (row_ok) {
          // 8 columns per 16-byte piece; pieces at or past the tensor's own
          // head dimension (D < 64 runs this kernel on zero-filled columns)
          // are not written.
          uint4* od = reinterpret_cast<uint4*>(row + col);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            if (col + 8 * v4 < p.D &&
                JVP_CHECK(col + 8 * v4 + 8 <= p.D && i < p.Nq, status, kChkGlobalCol))
              od[v4] = make_uint4(po[4 * v4], po[4 * v4 + 1], po[4 * v4 + 2], po[4 * v4 + 3]);
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------------
// Key-major kernel.  PART: 3 = all four key-side gradients (D = 64),
// 1 = value part (gV, g_dV), 2 = key part (gK, g_dK).
//
// TMEM: two score buffers of 128 columns (tile t uses buffer t & 1), each
// [S^T | dS^T] (value part, query tiles of BQ = 64 rows) or
// [S^T | dS^T | G^T | GP^T] (BQ = 32), then the accumulators from column 256.
// While the elementwise warps work on tile t, the score MMAs of tile t + 1
// fill the other buffer.  Shared memory: the resident key-side tiles, NS
// stages of query-side tiles, the stages' row scalars, the control block.
//
// PRIMAL (with PART = 3, at either D): the backward of attention without
// tangents.  A tile's buffer is [S^T | gP1^T] (BQ = 64 query rows, gP1 =
// gO V^T), the resident key-side tiles are K and V, a stage holds [Q] and
// [gO], and the accumulators are gV = P^T gO and gK = gS^T Q (2D columns, so
// one pass fits TMEM at D = 128 too).
template <int D, int PART, bool PRIMAL = false>
struct BkLayout {
  static constexpr bool kV = (PART & 1) != 0;
  static constexpr bool kK = (PART & 2) != 0;
  static constexpr int BK = 128;                          // keys per CTA
  static constexpr int NSC = (kK && !PRIMAL) ? 4 : 2;     // score matrices per tile
  static constexpr int BQ = 128 / NSC;    // query rows per tile (a buffer is 128 columns)
  static constexpr int KCH = D / 64;
  static constexpr int KT_BYTES = KCH * BK * 128;  // one [128 x D] key-side tile
  // [X rows | Y rows] of one 64-column chunk (primal: X rows alone)
  static constexpr int QCHUNK = (PRIMAL ? 1 : 2) * BQ * 128;
  static constexpr int QBLK = KCH * QCHUNK;        // a [X ; Y] block of one stage
  // key-side tiles resident for the whole CTA: K and dK always, V and dV for
  // the key part (primal: K and V)
  static constexpr int OFF_K = 0, OFF_DK = KT_BYTES;
  static constexpr int OFF_V = (PRIMAL ? 1 : 2) * KT_BYTES, OFF_DV = 3 * KT_BYTES;
  static constexpr int KSIDE = (PRIMAL ? 2 : kK ? 4 : 2) * KT_BYTES;
  // per stage: [Q ; dQ] and [gtO ; gO]; the row scalars (a float4 per query
  // row) of each stage live in a separate array so stages stay 1 KB aligned
  static constexpr int STAGE = 2 * QBLK;
  static constexpr int SCAL_BYTES = BQ * 16;
  static constexpr int CTRL_BYTES = 256;
  static constexpr int NS_FIT =
      (227 * 1024 - KSIDE - CTRL_BYTES - 1024) / (STAGE + SCAL_BYTES);
  static constexpr int NS = NS_FIT >= 4 ? 4 : NS_FIT;
  static constexpr int OFF_ST = KSIDE;
  static constexpr int OFF_SC = OFF_ST + NS * STAGE;
  static constexpr int OFF_CTRL = OFF_SC + NS * SCAL_BYTES;
  static constexpr int SMEM_BYTES = OFF_CTRL + CTRL_BYTES + 1024;
  static constexpr uint32_t TM_BUF = 128, TM_ACC = 256;
  static constexpr uint32_t S_OFF = 0, DS_OFF = BQ, G_OFF = 2 * BQ, GP_OFF = 3 * BQ;
  static_assert(NS >= 3 || D == 64 || !kK, "three stages for the key part");
  static_assert(NS >= 2, "two stages at least");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(D == 64 || PART != 3 || PRIMAL, "the four accumulators fit TMEM only at D = 64");
  static_assert(!PRIMAL || PART == 3, "the primal computes both key-side gradients in one pass");
  // Value part alone: the score products read only a stage's [Q ; dQ] half
  // and the accumulate products only its [gtO ; gO] half, so the two halves
  // have their own barriers and [Q ; dQ] is released (and refilled, one tile
  // ahead) as soon as the score products are done.
  static constexpr bool kSplitStage = kV && !kK;
};

template <int NS>
struct BwdKCtrl {
  uint64_t k_full;
  uint64_t q_full[NS], q_empty[NS];
  uint64_t qq_full[NS], qq_empty[NS];  // the [Q ; dQ] half of a stage, when it has its own
  uint64_t s_full[2], p_full[2], o_full, drain;
  uint64_t acc_done[2], drain_acc;  // accumulate MMAs of the tile in each buffer are complete
  uint64_t drain_b;
  uint32_t tmem_base;
  int abort;
};

template <typename T, int D, int MASK, int PART, bool PRIMAL = false>
__global__ void __launch_bounds__(kBwdThreadsK, 1)
    bwd_k_tc_kernel(const __grid_constant__ BwdTcMaps maps, const BwdParams p, int group_heads,
                    unsigned int* status) {
  using L = BkLayout<D, PART, PRIMAL>;
  constexpr int NS = L::NS, BK = L::BK, BQ = L::BQ;
  constexpr bool kBF16 = ElemTraits<T>::kBF16;
  constexpr int KSD = D / 16;
  constexpr int KSQ = BQ / 16;
  constexpr uint32_t I_N2Q = idesc_f16(kBF16, 128, 2 * BQ, false);  // [X ; Y]^T score pairs
  constexpr uint32_t I_NQ = idesc_f16(kBF16, 128, BQ, false);
  constexpr uint32_t I_ACC2 = idesc_f16(kBF16, 128, 2 * D, true);
  constexpr uint32_t I_ACC1 = idesc_f16(kBF16, 128, D, true);
  // Accumulator columns (relative to TM_ACC)
  constexpr uint32_t A_GDV = 0, A_GV = PRIMAL ? 0 : D;              // value part
  constexpr uint32_t A_GDK = L::kV ? 2 * D : 0;                      // key part
  constexpr uint32_t A_GK = PRIMAL ? D : A_GDK + D;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  static_assert(sizeof(BwdKCtrl<NS>) <= L::CTRL_BYTES, "control block budget");
  BwdKCtrl<NS>* ctrl = reinterpret_cast<BwdKCtrl<NS>*>(smem + L::OFF_CTRL);
  volatile int* abort = &ctrl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // One CTA per (batch, key/value head, key tile); with grouped-query
  // attention it visits the query tiles of every query head of its group.
  const int Hkv = p.H / p.kv_group;
  const int BH = p.B * Hkv;
  const int nk = (p.Nk + BK - 1) / BK;
  const int G = group_heads;
  // Key-major split: the ksplits CTAs of one key tile are adjacent.
  const int KS = p.ksplits > 1 ? p.ksplits : 1;
  const int split = static_cast<int>(blockIdx.x % KS);
  const int item = static_cast<int>(blockIdx.x / KS);
  const int g = item / (G * nk);
  const int rem = item - g * G * nk;
  const int Gg = min(G, BH - g * G);
  const int k_rank = rem / Gg;
  const int bhk = g * G + rem % Gg;
  const int kt = k_rank;  // causal: the first key tiles see the most query rows
  const int b = bhk / Hkv, hk = bhk % Hkv;
  const int j0 = kt * BK;
  const int nqt = (p.Nq + BQ - 1) / BQ;
  const bool causal =
      (MASK == kMaskCausal) || ((MASK == kMaskBool || MASK == kMaskAdditive) && p.causal != 0);
  const int t_begin = causal ? min(j0 / BQ, nqt) : 0;  // rows i >= j0 only
  const int n_th = nqt - t_begin;                       // query tiles per query head
  const int n_all = n_th * p.kv_group;                  // tiles over the whole group
  // This CTA's tiles [t_lo, t_lo + n_t) of the group's (all of them unless split)
  const int per_split = (n_all + KS - 1) / KS;
  const int t_lo = min(n_all, split * per_split);
  const int n_t = min(n_all, t_lo + per_split) - t_lo;

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->k_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctrl->q_full[s], 2);  // TMA bytes + the row scalars written by warp 0
      mbar_init(&ctrl->q_empty[s], 1);
      mbar_init(&ctrl->qq_full[s], 1);
      mbar_init(&ctrl->qq_empty[s], 1);
    }
    for (int u = 0; u < 2; ++u) {
      // key part: one commit from each of the two score-issuing threads
      mbar_init(&ctrl->s_full[u], L::kK ? 2 : 1);
      mbar_init(&ctrl->p_full[u], 256);
      mbar_init(&ctrl->acc_done[u], 1);
    }
    mbar_init(&ctrl->o_full, 1);
    mbar_init(&ctrl->drain, 1);
    mbar_init(&ctrl->drain_acc, 1);
    mbar_init(&ctrl->drain_b, 1);
    ctrl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues the TMA copies; all 32 lanes then write the stage's row
    // scalars (lse * log2 e, mu, nu, delta per query row; rows past Nq get
    // lse = -inf) and lane 0 adds the second arrival on q_full.
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctrl->k_full, L::KSIDE);
      for (int c = 0; c < L::KCH; ++c) {
        const int o = c * BK * 128;
        tma_load_4d(smem + L::OFF_K + o, &maps.k, &ctrl->k_full, c * 64, j0, hk, b);
        if (PRIMAL) {
          tma_load_4d(smem + L::OFF_V + o, &maps.v, &ctrl->k_full, c * 64, j0, hk, b);
        } else {
          tma_load_4d(smem + L::OFF_DK + o, &maps.dk, &ctrl->k_full, c * 64, j0, hk, b);
          if (L::kK) {
            tma_load_4d(smem + L::OFF_V + o, &maps.v, &ctrl->k_full, c * 64, j0, hk, b);
            tma_load_4d(smem + L::OFF_DV + o, &maps.dv, &ctrl->k_full, c * 64, j0, hk, b);
          }
        }
      }
    }
    // Row scalars of tile t for this lane's rows (lane + 32 u): the loads for
    // tile t + 1 are issued right after tile t's are published, so their
    // latency overlaps the wait for the next free stage.
    constexpr int RPL = BQ / 32;  // query rows per producer lane
    const CUtensorMap* mq = BQ == 64 ? &maps.q64 : &maps.q;
    const CUtensorMap* mdq = BQ == 64 ? &maps.dq64 : &maps.dq;
    const CUtensorMap* mgo = BQ == 64 ? &maps.go64 : &maps.go;
    const CUtensorMap* mgto = BQ == 64 ? &maps.gto64 : &maps.gto;
    float4 next[RPL];
    auto load_scalars = [&](int t) {
      const int h = hk * p.kv_group + (t_lo + t) / n_th;
#pragma unroll
      for (int u = 0; u < RPL; ++u) {
        const int i = (t_begin + (t_lo + t) % n_th) * BQ + lane + 32 * u;
        float4 v = make_float4(-INFINITY, 0.f, 0.f, 0.f);
        if (i < p.Nq && JVP_CHECK(h < p.H, status, kChkGlobalRow)) {
          const long long idx = (static_cast<long long>(b) * p.H + h) * p.Nq + i;
          v.x = p.lse[idx] * kLog2e;
          if (!PRIMAL) v.y = p.mu[idx];
          if (L::kK) {
            if (!PRIMAL) v.z = p.nu[idx];
            v.w = p.delta[idx];
          }
        }
        next[u] = v;
      }
    };
    if (n_t > 0) load_scalars(0);
    int fills = 0, qfills = 0;
    // The [Q ; dQ] half of tile tq's stage on its own barriers (lane 0).
    auto load_q = [&](int tq) -> bool {
      const int sq = tq % NS;
      if (!mbar_wait(&ctrl->qq_empty[sq], ((tq / NS) & 1) ^ 1, abort)) return false;
      const int hq = hk * p.kv_group + (t_lo + tq) / n_th;
      const int iq = (t_begin + (t_lo + tq) % n_th) * BQ;
      uint8_t* stq = smem + L::OFF_ST + sq * L::STAGE;
      mbar_arrive_expect_tx(&ctrl->qq_full[sq], L::QBLK);
      for (int c = 0; c < L::KCH; ++c) {
        tma_load_4d(stq + c * L::QCHUNK, mq, &ctrl->qq_full[sq], c * 64, iq, hq, b);
        tma_load_4d(stq + c * L::QCHUNK + BQ * 128, mdq, &ctrl->qq_full[sq], c * 64, iq, hq, b);
      }
      ++qfills;
      return true;
    };
    bool q_ok = true;
    if (L::kSplitStage && n_t > 0 && lane == 0) q_ok = load_q(0);
    q_ok = __shfl_sync(0xffffffffu, q_ok, 0);  // warp-uniform loop condition
    if (!q_ok && lane == 0) record_timeout(status, abort);
    for (int t = 0; q_ok && t < n_t; ++t) {
      const int s = t % NS;
      const uint32_t ph = (t / NS) & 1;
      const int h = hk * p.kv_group + (t_lo + t) / n_th;  // query head of this tile
      const int i0 = (t_begin + (t_lo + t) % n_th) * BQ;
      bool got = true;
      if (lane == 0) {
        if (L::kSplitStage && t + 1 < n_t) got = load_q(t + 1);
        if (got) got = mbar_wait(&ctrl->q_empty[s], ph ^ 1, abort);
      }
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        if (lane == 0) record_timeout(status, abort);
        break;
      }
      uint8_t* st = smem + L::OFF_ST + s * L::STAGE;
      if (lane == 0) {
        if constexpr (L::kSplitStage) {
          mbar_arrive_expect_tx(&ctrl->q_full[s], L::QBLK);
        } else {
          mbar_arrive_expect_tx(&ctrl->q_full[s], 2 * L::QBLK);
        }
        for (int c = 0; c < L::KCH; ++c) {
          if (PRIMAL) {  // [Q] then [gO]
            tma_load_4d(st + c * L::QCHUNK, mq, &ctrl->q_full[s], c * 64, i0, h, b);
            tma_load_4d(st + L::QBLK + c * L::QCHUNK, mgo, &ctrl->q_full[s], c * 64, i0, h, b);
            continue;
          }
          if (!L::kSplitStage) {
            tma_load_4d(st + c * L::QCHUNK, mq, &ctrl->q_full[s], c * 64, i0, h, b);
            tma_load_4d(st + c * L::QCHUNK + BQ * 128, mdq, &ctrl->q_full[s], c * 64, i0, h, b);
          }
          tma_load_4d(st + L::QBLK + c * L::QCHUNK, mgto, &ctrl->q_full[s], c * 64, i0, h, b);
          tma_load_4d(st + L::QBLK + c * L::QCHUNK + BQ * 128, mgo, &ctrl->q_full[s], c * 64, i0,
                      h, b);
        }
      }
#pragma unroll
      for (int u = 0; u < RPL; ++u)
        reinterpret_cast<float4*>(smem + L::OFF_SC + s * L::SCAL_BYTES)[lane + 32 * u] = next[u];
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->q_full[s]);
      ++fills;
      if (t + 1 < n_t) load_scalars(t + 1);
    }
    if (lane == 0 && *abort) {
      const int zero = 0;
      mbar_wait(&ctrl->k_full, 0, &zero);
      for (int t = max(0, fills - NS); t < fills; ++t)
        mbar_wait(&ctrl->q_full[t % NS], (t / NS) & 1, &zero);
      for (int t = max(0, qfills - NS); t < qfills; ++t)
        mbar_wait(&ctrl->qq_full[t % NS], (t / NS) & 1, &zero);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ score MMAs
    if (lane == 0) {
      bool ok = mbar_wait(&ctrl->k_full, 0, abort);
      tc_fence_after();
      const uint32_t aK = smem_u32(smem + L::OFF_K), adK = smem_u32(smem + L::OFF_DK);

      // Score products of tile t into buffer t & 1 (the key part's second
      // group, [G^T | V gO^T] and its dV gtO^T term, is issued by warp 11).
      auto issue_scores = [&](int t) -> bool {
        const int s = t % NS;
        if (!mbar_wait(L::kSplitStage ? &ctrl->qq_full[s] : &ctrl->q_full[s], (t / NS) & 1, abort))
          return false;
        tc_fence_after();
        const uint32_t qb = smem_u32(smem + L::OFF_ST + s * L::STAGE);  // [Q ; dQ]
        const uint32_t buf = tmem + (t & 1) * L::TM_BUF;
#pragma unroll
        for (int kk = 0; kk < KSD; ++kk) {  // [S^T | K dQ^T] = K [Q ; dQ]^T  (primal: S^T = K Q^T)
          const uint32_t off = (kk & 3) * 32;
          mma_ss(buf + L::S_OFF, sdesc_sw128(aK + (kk >> 2) * BK * 128 + off, 16, 1024),
                 sdesc_sw128(qb + (kk >> 2) * L::QCHUNK + off, 16, 1024),
                 PRIMAL ? I_NQ : I_N2Q, kk > 0);
        }
        if (!PRIMAL) {
#pragma unroll
          for (int kk = 0; kk < KSD; ++kk) {  // K dQ^T += dK Q^T  (= dS_raw^T)
            const uint32_t off = (kk & 3) * 32;
            mma_ss(buf + L::DS_OFF, sdesc_sw128(adK + (kk >> 2) * BK * 128 + off, 16, 1024),
                   sdesc_sw128(qb + (kk >> 2) * L::QCHUNK + off, 16, 1024), I_NQ, 1u);
          }
        }
        if (L::kSplitStage) mma_commit(&ctrl->qq_empty[s]);
        mma_commit(&ctrl->s_full[t & 1]);
        return true;
      };

      // Tile t's scores go into buffer t & 1 once its stage has landed and the
      // accumulate MMAs of tile t - 2 (the buffer's previous reader) are done.
      for (int t = 0; ok && t < n_t; ++t) {
        if (t >= 2 && !mbar_wait(&ctrl->acc_done[t & 1], ((t - 2) >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        if (!issue_scores(t)) {
          ok = false;
          break;
        }
      }
      if (!ok) record_timeout(status, abort);
      mma_commit(&ctrl->drain);
      const int zero = 0;
      mbar_wait(&ctrl->drain, 0, &zero);
    }
  } else if (warp == kBwdAccWarp) {
    // ------------------------------------------------------------ accumulate MMAs
    if (lane == 0) {
      bool ok = true;
      for (int t = 0; ok && t < n_t; ++t) {
        if (!mbar_wait(&ctrl->p_full[t & 1], (t >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int s = t % NS;
        const uint32_t qb = smem_u32(smem + L::OFF_ST + s * L::STAGE);
        const uint32_t ob = qb + L::QBLK;
        const uint32_t buf = tmem + (t & 1) * L::TM_BUF;
        // A operands of query rows [16 kk, 16 kk + 16) of the tile: P^T at
        // buffer column 16 kk (dP^T at + 8), gS^T at DS_OFF + 16 kk (g_dS^T at + 8).
        if constexpr (PRIMAL) {
          // gV += P^T gO ; gK += gS^T Q  (P^T at buffer column 16 kk, gS^T at
          // DS_OFF + 16 kk; [Q] and [gO] chunks QCHUNK apart)
#pragma unroll
          for (int kk = 0; kk < KSQ; ++kk) {
            const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + L::TM_ACC + A_GV, buf + kk * 16,
                   sdesc_sw128(ob + kk * 16 * 128, L::QCHUNK, 1024), I_ACC1, acc);
            mma_ts(tmem + L::TM_ACC + A_GK, buf + L::DS_OFF + kk * 16,
                   sdesc_sw128(qb + kk * 16 * 128, L::QCHUNK, 1024), I_ACC1, acc);
          }
        }
#pragma unroll
        for (int kk = 0; kk < KSQ && !PRIMAL; ++kk) {
          const uint32_t a0 = buf + kk * 16;
          const uint32_t ag = buf + L::DS_OFF + kk * 16;
          const uint32_t xq = qb + kk * 16 * 128;  // MN-major: 16 query rows per K-step
          const uint32_t xo = ob + kk * 16 * 128;
          const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
          if (L::kV) {
            if (D == 64) {  // [g_dV | gV] += P^T [gtO | gO]
              mma_ts(tmem + L::TM_ACC + A_GDV, a0, sdesc_sw128(xo, BQ * 128, 1024), I_ACC2, acc);
            } else {
              mma_ts(tmem + L::TM_ACC + A_GDV, a0, sdesc_sw128(xo, L::QCHUNK, 1024), I_ACC1, acc);
              mma_ts(tmem + L::TM_ACC + A_GV, a0, sdesc_sw128(xo + BQ * 128, L::QCHUNK, 1024),
                     I_ACC1, acc);
            }
          }
          if (L::kK) {
            if (D == 64) {  // [g_dK | gK] += g_dS^T [Q | dQ]
              mma_ts(tmem + L::TM_ACC + A_GDK, ag + 8, sdesc_sw128(xq, BQ * 128, 1024), I_ACC2,
                     acc);
            } else {
              mma_ts(tmem + L::TM_ACC + A_GDK, ag + 8, sdesc_sw128(xq, L::QCHUNK, 1024), I_ACC1,
                     acc);
              mma_ts(tmem + L::TM_ACC + A_GK, ag + 8, sdesc_sw128(xq + BQ * 128, L::QCHUNK, 1024),
                     I_ACC1, acc);
            }
          }
        }
#pragma unroll
        for (int kk = 0; kk < KSQ && !PRIMAL; ++kk) {
          const uint32_t a0 = buf + kk * 16;
          const uint32_t ag = buf + L::DS_OFF + kk * 16;
          if (L::kV)  // gV += dP^T gtO
            mma_ts(tmem + L::TM_ACC + A_GV, a0 + 8,
                   sdesc_sw128(ob + kk * 16 * 128, D == 64 ? BQ * 128 : L::QCHUNK, 1024), I_ACC1,
                   1u);
          if (L::kK)  // gK += gS^T Q
            mma_ts(tmem + L::TM_ACC + A_GK, ag,
                   sdesc_sw128(qb + kk * 16 * 128, D == 64 ? BQ * 128 : L::QCHUNK, 1024), I_ACC1,
                   1u);
        }
        mma_commit(&ctrl->q_empty[s]);
        mma_commit(&ctrl->acc_done[t & 1]);
      }
      if (ok && n_t > 0) mma_commit(&ctrl->o_full);
      if (!ok) record_timeout(status, abort);
      mma_commit(&ctrl->drain_acc);
      const int zero = 0;
      mbar_wait(&ctrl->drain_acc, 0, &zero);
    }
  } else if (warp == kBwdScoreWarpB) {
    // ------------------------------------------------------------ score MMAs, group B
    // Key part: [G^T | V gO^T] = V [gtO ; gO]^T and V gO^T += dV gtO^T write
    // columns [G_OFF, G_OFF + 2 BQ) of the buffer, disjoint from warp 1's
    // products, so the two groups are issued side by side.  Same buffer rule:
    // tile t waits for its stage and for the accumulate MMAs of tile t - 2.
    if (L::kK && lane == 0) {
      bool ok = mbar_wait(&ctrl->k_full, 0, abort);
      tc_fence_after();
      const uint32_t aV = smem_u32(smem + L::OFF_V), adV = smem_u32(smem + L::OFF_DV);
      for (int t = 0; ok && t < n_t; ++t) {
        const int s = t % NS;
        if ((t >= 2 && !mbar_wait(&ctrl->acc_done[t & 1], ((t - 2) >> 1) & 1, abort)) ||
            !mbar_wait(&ctrl->q_full[s], (t / NS) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ob = smem_u32(smem + L::OFF_ST + s * L::STAGE) + L::QBLK;  // [gtO ; gO]
        const uint32_t buf = tmem + (t & 1) * L::TM_BUF;
        if (PRIMAL) {
#pragma unroll
          for (int kk = 0; kk < KSD; ++kk) {  // gP1^T = V gO^T
            const uint32_t off = (kk & 3) * 32;
            mma_ss(buf + L::DS_OFF, sdesc_sw128(aV + (kk >> 2) * BK * 128 + off, 16, 1024),
                   sdesc_sw128(ob + (kk >> 2) * L::QCHUNK + off, 16, 1024), I_NQ, kk > 0);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < KSD; ++kk) {  // [G^T | V gO^T] = V [gtO ; gO]^T
            const uint32_t off = (kk & 3) * 32;
            mma_ss(buf + L::G_OFF, sdesc_sw128(aV + (kk >> 2) * BK * 128 + off, 16, 1024),
                   sdesc_sw128(ob + (kk >> 2) * L::QCHUNK + off, 16, 1024), I_N2Q, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < KSD; ++kk) {  // V gO^T += dV gtO^T  (= gP1^T)
            const uint32_t off = (kk & 3) * 32;
            mma_ss(buf + L::GP_OFF, sdesc_sw128(adV + (kk >> 2) * BK * 128 + off, 16, 1024),
                   sdesc_sw128(ob + (kk >> 2) * L::QCHUNK + off, 16, 1024), I_NQ, 1u);
          }
        }
        mma_commit(&ctrl->s_full[t & 1]);
      }
      if (!ok) record_timeout(status, abort);
      mma_commit(&ctrl->drain_b);
      const int zero = 0;
      mbar_wait(&ctrl->drain_b, 0, &zero);
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ elementwise
    // Thread = key (TMEM lane); warpgroup wg owns query rows [wg*QW, wg*QW + QW)
    // of every tile, taken 16 at a time.
    constexpr int QW = BQ / 2;
    const int wg = (warp - 2) >> 2;
    const int sub = warp & 3;
    const int r = sub * 32 + lane;
    const int j = j0 + r;
    const bool key_ok = j < p.Nk;
    const uint32_t lb = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const float c = p.scale * kLog2e;
    const float s = p.scale;
    bool ok = true;
    for (int t = 0; t < n_t; ++t) {
      const int st_i = t % NS;
      const int h = hk * p.kv_group + (t_lo + t) / n_th;            // query head of this tile
      const int i0 = (t_begin + (t_lo + t) % n_th) * BQ + wg * QW;  // first query row of this warpgroup
      // This thread's key's mask entries for the warpgroup's QW rows, requested
      // before the wait for the tile's scores so that their latency overlaps it
      // (rows past Nq read row Nq - 1 and are not used).
      MaskCol<MASK, QW> mcv;
      if constexpr (MASK == kMaskBool || MASK == kMaskAdditive) {
        const long long mcol = static_cast<long long>(b) * p.msb +
                               static_cast<long long>(h) * p.msh +
                               static_cast<long long>(key_ok ? j : 0) * p.msk;
#pragma unroll
        for (int q = 0; q < QW; ++q)
          mcv.load(q, p.mask, mcol + static_cast<long long>(min(i0 + q, p.Nq - 1)) * p.msq);
      }
      if (!warp_wait(&ctrl->s_full[t & 1], (t >> 1) & 1, status, abort) ||
          !warp_wait(&ctrl->q_full[st_i], (t / NS) & 1, status, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4* rsc =
          reinterpret_cast<const float4*>(smem + L::OFF_SC + st_i * L::SCAL_BYTES) + wg * QW;
      const uint32_t bcol = (t & 1) * L::TM_BUF + wg * QW;
#pragma unroll
      for (int hq = 0; hq < QW / 16; ++hq) {
        // The 16-bit results go only into the 16 columns this half has just
        // read (S^T at col, dS^T at DS_OFF + col), so the other halves' inputs stay intact.
        const uint32_t col = bcol + hq * 16;
        uint32_t rs[16], rds[16], rg[16], rgp[16];
        const uint32_t top = (L::kK && !PRIMAL) ? L::GP_OFF : L::DS_OFF;
        const bool cols_ok = JVP_CHECK(col + top + 16 <= 512u && col + L::DS_OFF + 16 <= 512u &&
                                           wg * QW + hq * 16 + 16 <= L::SCAL_BYTES / 16,
                                       status, kChkTmem);
        if (PRIMAL) {  // S^T and gP1^T; dS = G = 0
#pragma unroll
          for (int e = 0; e < 16; ++e) rds[e] = rg[e] = 0u;
          if (cols_ok) tmem_ld16x2(lb + col + L::S_OFF, lb + col + L::DS_OFF, rs, rgp);
        } else if (cols_ok) {
          tmem_ld16x2(lb + col + L::S_OFF, lb + col + L::DS_OFF, rs, rds);
          if (L::kK) tmem_ld16x2(lb + col + L::G_OFF, lb + col + L::GP_OFF, rg, rgp);
        }
        uint32_t pa[8], pb[8], pc[8], pd[8];  // P^T, dP^T, gS^T, g_dS^T (packed pairs)
#pragma unroll
        for (int qq = 0; qq < 16; qq += 2) {
          float P2[2], dP2[2], gS2[2], gdS2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = i0 + hq * 16 + qq + e;
            const float4 rv = rsc[hq * 16 + qq + e];  // lse2, mu, nu, delta (one broadcast read)
            bool keep = key_ok && rv.x != -INFINITY;  // false for rows past Nq
            float x = fmaf(__uint_as_float(rs[qq + e]), c, -rv.x);
            if (causal) keep = keep && j <= i;
            if constexpr (MASK == kMaskBool) keep = keep && mcv.keep(hq * 16 + qq + e);
            if constexpr (MASK == kMaskAdditive) {
              x = fmaf(keep ? mcv.add(hq * 16 + qq + e) : 0.f, kLog2e, x);
              keep = keep && x != -INFINITY;
            }
            const float gv = L::kK ? __uint_as_float(rg[qq + e]) : 0.f;
            const float gp = L::kK ? __uint_as_float(rgp[qq + e]) : 0.f;
            const BwdTerms bt =
                bwd_terms(keep, x, __uint_as_float(rds[qq + e]), gv, gp, s, rv.y, rv.z, rv.w);
            P2[e] = bt.P;
            dP2[e] = bt.dP;
            gS2[e] = bt.gS;
            gdS2[e] = bt.gdS;
          }
          pa[qq >> 1] = ElemTraits<T>::pack(P2[0], P2[1]);
          pb[qq >> 1] = ElemTraits<T>::pack(dP2[0], dP2[1]);
          pc[qq >> 1] = ElemTraits<T>::pack(gS2[0], gS2[1]);
          pd[qq >> 1] = ElemTraits<T>::pack(gdS2[0], gdS2[1]);
        }
        if (L::kV && cols_ok) {
          tmem_st8(lb + col + L::S_OFF, pa);
          if (!PRIMAL) tmem_st8(lb + col + L::S_OFF + 8, pb);
        }
        if (L::kK && cols_ok) {
          tmem_st8(lb + col + L::DS_OFF, pc);
          if (!PRIMAL) tmem_st8(lb + col + L::DS_OFF + 8, pd);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctrl->p_full[t & 1]);
    }
    if (ok && n_t > 0) ok = warp_wait(&ctrl->o_full, 0, status, abort);
    if (ok) {
      tc_fence_after();
      // Output tensors of this kernel, split between the two warpgroups.
      constexpr int NOUT = PRIMAL ? 2 : (L::kV ? 2 : 0) + (L::kK ? 2 : 0);
#pragma unroll 1
      for (int oi = wg; oi < NOUT; oi += 2) {
        // oi enumerates g_dV, gV (value part) then g_dK, gK (key part); the
        // primal's are gV and gK
        const int which = PRIMAL ? 2 * oi + 1 : L::kV ? oi : oi + 2;
        void* dst = which == 0 ? p.g_dv : which == 1 ? p.g_v : which == 2 ? p.g_dk : p.g_k;
        const Strides& ds = which == 0 ? p.sgdv : which == 1 ? p.sgv : which == 2 ? p.sgdk : p.sgk;
        const uint32_t acol = which == 0 ? A_GDV : which == 1 ? A_GV : which == 2 ? A_GDK : A_GK;
        const float scl = which >= 2 ? s : 1.0f;
        T* row = static_cast<T*>(dst) + static_cast<long long>(b) * ds.b +
                 static_cast<long long>(hk) * ds.h + static_cast<long long>(key_ok ? j : 0) * ds.n;
        // split: this CTA's fp32 partial row of the gradient
        float* prow = p.kws + ((static_cast<long long>(split) * 4 + which) * BH + bhk) *
                                  static_cast<long long>(p.Nk) * D +
                      static_cast<long long>(key_ok ? j : 0) * D;
#pragma unroll 1
        for (int col = 0; col < D; col += 32) {
          uint32_t a[32];
          if (n_t > 0 && JVP_CHECK(L::TM_ACC + acol + col + 32 <= 512u, status, kChkTmem)) {
            tmem_ld32(lb + L::TM_ACC + acol + col, a);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = 0u;
          }
          if (KS > 1) {
            if (key_ok && JVP_CHECK(j < p.Nk, status, kChkGlobalCol)) {
              float4* pd = reinterpret_cast<float4*>(prow + col);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                pd[v4] = make_float4(__uint_as_float(a[4 * v4]) * scl,
                                     __uint_as_float(a[4 * v4 + 1]) * scl,
                                     __uint_as_float(a[4 * v4 + 2]) * scl,
                                     __uint_as_float(a[4 * v4 + 3]) * scl);
            }
            continue;
          }
          uint32_t po[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            po[e >> 1] =
                ElemTraits<T>::pack(__uint_as_float(a[e]) * scl, __uint_as_float(a[e + 1]) * scl);
          if (key_ok) {
            uint4* od = reinterpret_cast<uint4*>(row + col);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              if (col + 8 * v4 < p.D &&  // (see the query-major kernel's store)
                  JVP_CHECK(col + 8 * v4 + 8 <= p.D && j < p.Nk, status, kChkGlobalCol))
                od[v4] = make_uint4(po[4 * v4], po[4 * v4 + 1], po[4 * v4 + 2], po[4 * v4 + 3]);
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Query-major split: adds the qsplits fp32 partial sums of g_dQ (slot 0, when
// bit 0 of which_mask) and gQ (slot 1, bit 1) into the outputs' dtype, D real
// columns.  One thread per four columns of one row.
template <typename T, int DK>
__global__ void bwd_query_combine_kernel(const BwdParams p, int which_mask) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  constexpr int kPieces = DK / 4;
  const long long n = 2 * rows * kPieces;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int which = static_cast<int>(idx / (rows * kPieces));
    const long long rr = (idx / kPieces) % rows;
    const int c = static_cast<int>(idx % kPieces) * 4;
    if (!((which_mask >> which) & 1) || c >= p.D) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < p.qsplits; ++sp) {
      const float4 v = *reinterpret_cast<const float4*>(
          p.qws + ((static_cast<long long>(sp) * 2 + which) * rows + rr) * DK + c);
      acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    const long long bh = rr / p.Nq, i = rr % p.Nq;
    const long long b = bh / p.H, h = bh % p.H;
    void* dst = which == 0 ? p.g_dq : p.g_q;
    const Strides& ds = which == 0 ? p.sgdq : p.sgq;
    T* o = static_cast<T*>(dst) + b * ds.b + h * ds.h + i * ds.n + c;
    *reinterpret_cast<uint2*>(o) =
        make_uint2(ElemTraits<T>::pack(acc.x, acc.y), ElemTraits<T>::pack(acc.z, acc.w));
  }
}

// Key-major split: adds the ksplits fp32 partial sums of each key-side
// gradient in `which_mask` (bit w: 0 g_dV, 1 gV, 2 g_dK, 3 gK) and writes the
// result, in the outputs' dtype, to the D real columns.  One thread per four
// columns of one row of one gradient.
template <typename T, int DK>
__global__ void bwd_key_combine_kernel(const BwdParams p, int which_mask) {
  const int Hkv = p.H / p.kv_group;
  const long long rows = static_cast<long long>(p.B) * Hkv * p.Nk;
  constexpr int kPieces = DK / 4;
  const long long n = 4 * rows * kPieces;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int which = static_cast<int>(idx / (rows * kPieces));
    const long long rr = (idx / kPieces) % rows;
    const int c = static_cast<int>(idx % kPieces) * 4;
    if (!((which_mask >> which) & 1) || c >= p.D) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < p.ksplits; ++sp) {
      const float4 v = *reinterpret_cast<const float4*>(
          p.kws + ((static_cast<long long>(sp) * 4 + which) * rows + rr) * DK + c);
      acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    const long long bhk = rr / p.Nk, jk = rr % p.Nk;
    const long long b = bhk / Hkv, hk = bhk % Hkv;
    void* dst = which == 0 ? p.g_dv : which == 1 ? p.g_v : which == 2 ? p.g_dk : p.g_k;
    const Strides& ds = which == 0 ? p.sgdv : which == 1 ? p.sgv : which == 2 ? p.sgdk : p.sgk;
    T* o = static_cast<T*>(dst) + b * ds.b + hk * ds.h + jk * ds.n + c;
    *reinterpret_cast<uint2*>(o) =
        make_uint2(ElemTraits<T>::pack(acc.x, acc.y), ElemTraits<T>::pack(acc.z, acc.w));
  }
}

// ----------------------------------------------------------------------------
// Launch of the tensor-core backward (after the row pre-pass).
// Keyed on the kernel itself (all backward kernels share one signature), so
// each kernel gets its own per-device record of the attribute being set.
template <auto kern>
cudaError_t set_smem(int bytes) {
  static std::atomic<unsigned long long> done{0};  // per device; shared by host threads
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && (done.load(std::memory_order_relaxed) & (1ull << dev))) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done.fetch_or(1ull << dev, std::memory_order_relaxed);
  return e;
}

// qmaps: query-major kernel (query side 128-row boxes, key side 64); kmaps:
// key-major kernel (key side 128-row boxes, query side 32, and 64 in q64 ...).
// The query-major kernel on `stream`, the key-major kernel(s) on `kstream`.
template <typename T, int D, int MASK, bool PRIMAL>
cudaError_t launch_bwd_tc_variant(const BwdTcMaps& qmaps, const BwdTcMaps& kmaps,
                                  const BwdParams& p, int num_sms, unsigned int* status,
                                  cudaStream_t stream, cudaStream_t kstream) {
  const int BH = p.B * p.H;
  {
    using L = BqLayout<D, PRIMAL>;
    constexpr auto kern = bwd_q_tc_kernel<T, D, MASK, PRIMAL>;
    cudaError_t e = set_smem<kern>(L::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int nq = (p.Nq + L::BM - 1) / L::BM;
    // About one wave of CTAs per group of heads; causal problems (their tiles
    // run longest first within a group) take as many heads as keep the key
    // side's tiles within 32 MB of L2, which shortens the launch's tail.
    int G = max(1, min(BH, num_sms / max(1, nq)));
    if (MASK == kMaskCausal || p.causal) {
      const double kv_head = (PRIMAL ? 2.0 : 4.0) * static_cast<double>(p.Nk) * D * sizeof(T);
      G = max(G, min(BH, static_cast<int>(32.0 * 1048576.0 / kv_head)));
    }
    const int QS = p.qsplits > 1 ? p.qsplits : 1;
    kern<<<static_cast<unsigned>(static_cast<long long>(nq) * BH * QS), kBwdThreads,
           L::SMEM_BYTES, stream>>>(qmaps, p, G, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (QS > 1) {
      const long long n = 2LL * BH * p.Nq * (D / 4);
      const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 8LL * num_sms));
      bwd_query_combine_kernel<T, D><<<blocks, 256, 0, stream>>>(p, PRIMAL ? 0x2 : 0x3);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  auto key_side = [&](auto part_tag) -> cudaError_t {
    constexpr int PART = decltype(part_tag)::value;
    using L = BkLayout<D, PART, PRIMAL>;
    constexpr auto kern = bwd_k_tc_kernel<T, D, MASK, PART, PRIMAL>;
    cudaError_t e = set_smem<kern>(L::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int nk = (p.Nk + L::BK - 1) / L::BK;
    const int BHk = p.B * (p.H / p.kv_group);
    const int KS = p.ksplits > 1 ? p.ksplits : 1;
    int G = max(1, min(BHk, num_sms / max(1, nk)));
    if (MASK == kMaskCausal || p.causal) {  // as above, for the query side's tiles
      const double q_head =
          (PRIMAL ? 2.0 : 4.0) * static_cast<double>(p.Nq) * D * sizeof(T) * p.kv_group;
      G = max(G, min(BHk, static_cast<int>(32.0 * 1048576.0 / q_head)));
    }
    static_assert(L::BQ == 32 || L::BQ == 64, "query-side box heights of kmaps");
    kern<<<static_cast<unsigned>(static_cast<long long>(nk) * BHk * KS), kBwdThreadsK,
           L::SMEM_BYTES, kstream>>>(kmaps, p, G, status);
    return cudaGetLastError();
  };
  cudaError_t e;
  if constexpr (D == 64 || PRIMAL) {
    e = key_side(std::integral_constant<int, 3>{});
  } else {
    e = key_side(std::integral_constant<int, 1>{});
    if (e == cudaSuccess) e = key_side(std::integral_constant<int, 2>{});
  }
  if (e == cudaSuccess && p.ksplits > 1) {
    const long long n = 4LL * p.B * (p.H / p.kv_group) * p.Nk * (D / 4);
    const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 8LL * num_sms));
    bwd_key_combine_kernel<T, D><<<blocks, 256, 0, kstream>>>(p, PRIMAL ? 0xA : 0xF);
    e = cudaGetLastError();
  }
  return e;
}

template <typename T, int D, bool PRIMAL = false>
cudaError_t launch_bwd_tc_dispatch(int mask_kind, const BwdTcMaps& qmaps, const BwdTcMaps& kmaps,
                                   const BwdParams& p, int num_sms, unsigned int* status,
                                   cudaStream_t stream, cudaStream_t kstream) {
  switch (mask_kind) {
    case kMaskNone:
      return launch_bwd_tc_variant<T, D, kMaskNone, PRIMAL>(qmaps, kmaps, p, num_sms, status,
                                                            stream, kstream);
    case kMaskBool:
      return launch_bwd_tc_variant<T, D, kMaskBool, PRIMAL>(qmaps, kmaps, p, num_sms, status,
                                                            stream, kstream);
    case kMaskAdditive:
      return launch_bwd_tc_variant<T, D, kMaskAdditive, PRIMAL>(qmaps, kmaps, p, num_sms, status,
                                                                stream, kstream);
    case kMaskCausal:
      return launch_bwd_tc_variant<T, D, kMaskCausal, PRIMAL>(qmaps, kmaps, p, num_sms, status,
                                                              stream, kstream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace jvp

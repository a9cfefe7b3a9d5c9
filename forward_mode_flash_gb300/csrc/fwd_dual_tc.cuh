// fwd_dual_tc.cuh -- tensor-core (tcgen05 + TMEM + TMA) kernel for attention
// forward + JVP on sm_103a, fp16/bf16 inputs, fp32 accumulation.
//
// What it computes is the dual forward of softmax attention ("JVP Flash
// Attention" project page, Description and Usage sections):
//   S = s Q K^T + M,  P = softmax(S),  O = P V,
//   dS = s (dQ K^T + Q dK^T),  mu = rowsum(P * dS),
//   tO = (P * dS) V - mu O + P dV,  lse = log rowsum(exp S).
// It never materialises P or dS in global memory: one pass over key tiles
// keeps, per query row, a running maximum m, the row sum l = sum p~, the
// running sum mu~ = sum p~ * dS, and two TMEM accumulators
//   A = sum p~ V          T = sum p~ (dS V + dV)
// (p~ = exp(S - m)), then O = A / l, mu = mu~ / l, tO = T / l - mu O.
//
// Work decomposition: one CTA per (128-row query tile, batch*head), eleven
// warps (twelve or thirteen where more warps issue MMAs, see tc_threads), one
// CTA per SM (it owns all 512 TMEM columns).
//   warp 0      TMA producer: Q, dQ once; then per 64-key tile the [K;dK]
//               block and the [V|dV] block, through an NS-deep ring.
//   warp 1      TMEM allocator; one thread issues the score MMAs.
//   warps 2..9  softmax, two warpgroups: a thread owns one query row (its TMEM
//               lane) and one half (32 keys) of every key tile; the two halves
//               exchange their maxima through shared memory each tile.  The
//               epilogue splits the output columns the same way.
//   warp 10     one thread issues the P~V MMAs.
//   warps 11,12 (some variants) a second score and a second P~V issuing
//               thread, each taking the odd tiles.
// Per key tile t (buffer b = t % 2 of the double-buffered score region):
//   M1  [S | Q dK^T] = Q [K ; dK]^T          (N = 128, SMEM x SMEM)
//       -> S is final: the softmax starts (max, exchange, exponentials)
//   M2  Q dK^T      += dQ K^T                 (N = 64)
//   softmax: P~ written back to TMEM (16-bit) over the S columns, published;
//   M3  [A | T]     += P~ [V | dV]            (N = 2D, A operand from TMEM)
//   softmax, once M2 is done: P~ * s * dS_raw into its own dS columns
//   M4  T           += (P~ * dS) V            (N = D)
// M1/M2 of tile t+2 reuse buffer b once M3/M4 of tile t are done, so the
// tensor core computes the next scores while the softmax warps work.  (Without
// tangents there are four 64-column buffers, S alone, reused every 4 tiles;
// the softmax warpgroups then take whole tiles, and at D = 128 the score
// products come in pairs of tiles.)  The
// epilogue stages O and tO in the idle [K;dK] ring and writes them with TMA
// stores.
//
// Masks: a boolean keep-mask (and the additive mask at D = 64 or without
// tangents) is loaded into registers a tile ahead by each softmax thread for
// its own row.  At D = 128 with tangents an additive tile ahead does not fit
// the registers; when the mask's layout
// admits a tensor map (contiguous keys, rows that do not broadcast, 16-byte
// strides) the producer copies each [128 x 64] fp32 tile into a shared-memory
// slot a tile ahead, in two swizzled [128 x 32] boxes, and the softmax reads
// its row from there (else: per-row loads in the tile, the next tiles'
// lines prefetched into L2).  Room for the slot comes from the two [K;dK]
// stages sharing one dK slot (see TcLayout).
//
// Rescaling is conditional: the row maximum used in the exponent is only
// moved when a tile's maximum exceeds it by more than 2^8, so A, T, l and mu~
// are rarely touched; the final ratios are exact for any stale maximum.
//
// Consistent rounding: the tensor core consumes P~ and P~ * dS rounded to 16
// bits, so l and mu~ are summed from those same rounded values.  O and tO are
// then the exact attention output and JVP of a softmax whose weights are
// perturbed by one 16-bit rounding each, and the rounding errors enter tO
// multiplied by (V_j - O) rather than V_j (tO = T/l - mu O cancels).  A
// separate fp32 sum of the unrounded p~ gives the log-sum-exp.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "debug_checks.cuh"
#include "jvp_internal.h"
#include "sm103_ptx.cuh"

namespace jvp {

template <typename T>
struct ElemTraits;
template <>
struct ElemTraits<__half> {
  static constexpr bool kBF16 = false;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t x) {
    return __half22float2(*reinterpret_cast<__half2*>(&x));
  }
};
template <>
struct ElemTraits<__nv_bfloat16> {
  static constexpr bool kBF16 = true;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t x) {
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
  }
};

template <int D, bool TANGENT, bool MTILE = false>
struct TcLayout {
  static constexpr int BM = kTcBlockM;              // query rows per CTA
  static constexpr int BN = kTcBlockN;              // keys per tile
  static constexpr int KCH = D / 64;                // 128-byte chunks along D
  // K/V ring depth (three stages without tangents when two additive-mask
  // slots take the room of the fourth)
  static constexpr int NS = (D == 128 && TANGENT) ? 2 : (MTILE ? 3 : 4);
  // Score buffers in TMEM: with tangents two of 128 columns ([S | dS]);
  // without, four of 64 (S alone), so the score products can run up to three
  // tiles ahead of the softmax.
  static constexpr int NB = TANGENT ? 2 : 4;
  static constexpr uint32_t BUF_COLS = TANGENT ? 128 : 64;
  static constexpr int Q_BYTES = KCH * BM * 128;
  static constexpr int KROWS = TANGENT ? 2 * BN : BN;  // rows of the [K;dK] block
  static constexpr int KCHUNK_BYTES = KROWS * 128;     // one 64-column chunk of it
  static constexpr int KDK_BYTES = KCH * KCHUNK_BYTES;
  static constexpr int VCHUNK_BYTES = BN * 128;        // one 64-column chunk of V
  static constexpr int VDV_BYTES = (TANGENT ? 2 : 1) * KCH * VCHUNK_BYTES;
  // MTILE: the additive mask's [BM x BN] fp32 tile is brought into shared
  // memory by TMA a tile ahead (D = 128: one slot with tangents, where a tile
  // ahead does not fit the registers; two without, each thread's row loads
  // touching a line per row).  To make room next to the dual rings, the two [K;dK] stages
  // then share one dK slot: each 64-column chunk holds [K0 | dK | K1], stage 0
  // reads the 128 rows [K0; dK] and stage 1 the rows [dK; K1], so stage 1's
  // score products come out as [Q dK^T | S] instead of [S | Q dK^T].  The dK
  // slot is refilled once the first score product of a tile has read it.
  static constexpr bool kSharedDK = MTILE && TANGENT && NS == 2;
  static constexpr int KREGION = kSharedDK ? KCH * 3 * BN * 128 : NS * KDK_BYTES;
  static constexpr int NMS = MTILE ? (TANGENT ? 1 : 2) : 0;  // mask slots
  static constexpr int MSK_TILE = BM * BN * 4;                // one slot
  static constexpr int MSK_BYTES = NMS * MSK_TILE;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DQ = OFF_Q + Q_BYTES;
  static constexpr int OFF_KDK = OFF_DQ + (TANGENT ? Q_BYTES : 0);
  static constexpr int OFF_VDV = OFF_KDK + KREGION;
  static constexpr int OFF_MSK = OFF_VDV + NS * VDV_BYTES;
  static constexpr int OFF_CTRL = OFF_MSK + MSK_BYTES;
  // Without tangents the K ring is laid out chunk by chunk (chunk c of stage
  // s at (c * NS + s) * KCHUNK_BYTES), so that chunk c of stages s and s + 1
  // are 128 contiguous rows: one N = 128 score product covers two key tiles.
  static constexpr bool kChunkMajorK = !TANGENT;
  // Byte distance between the 64-column chunks of one stage's K rows.
  static constexpr int K_CHUNK_STRIDE =
      kSharedDK ? 3 * BN * 128 : kChunkMajorK ? NS * KCHUNK_BYTES : KCHUNK_BYTES;
  // Byte offsets of stage s, 64-column chunk c: the K rows, the dK rows, and
  // the first row of the 128-row operand of the first score product.
  static __device__ __forceinline__ int k_off(int s, int c) {
    return kSharedDK      ? OFF_KDK + c * 3 * BN * 128 + s * 2 * BN * 128
           : kChunkMajorK ? OFF_KDK + (c * NS + s) * KCHUNK_BYTES
                          : OFF_KDK + s * KDK_BYTES + c * KCHUNK_BYTES;
  }
  static __device__ __forceinline__ int dk_off(int s, int c) {
    return kSharedDK ? OFF_KDK + c * 3 * BN * 128 + BN * 128 : k_off(s, c) + BN * 128;
  }
  static __device__ __forceinline__ int m1_off(int s, int c) {
    return kSharedDK ? OFF_KDK + c * 3 * BN * 128 + s * BN * 128 : k_off(s, c);
  }
  // TMEM columns of S and of dS in score buffer buf (stage buf; NS = 2 when
  // the dK slot is shared, so the stage of a tile is its buffer).
  static __device__ __forceinline__ uint32_t buf_col(int buf) {
    return static_cast<uint32_t>(buf) * BUF_COLS;
  }
  static __device__ __forceinline__ uint32_t s_col(int buf) {
    return buf_col(buf) + ((kSharedDK && buf) ? BN : 0);
  }
  static __device__ __forceinline__ uint32_t ds_col(int buf) {
    return buf_col(buf) + ((kSharedDK && buf) ? 0 : BN);
  }
  static constexpr int CTRL_BYTES = 8192;
  static constexpr int USED = OFF_CTRL + CTRL_BYTES;
  // Padded so that only one CTA fits per SM (each CTA owns all 512 TMEM columns).
  static constexpr int SMEM_BYTES = (USED + 1024 < 120 * 1024 ? 120 * 1024 : USED + 1024);
  // TMEM columns.  At D = 64, and without tangents at D = 128 too, each
  // softmax warpgroup keeps its own running max, sums and [A | T] (or A)
  // accumulator for its half of every key tile (the two accumulators fit next
  // to the score buffers), so no per-tile exchange of half-row maxima is
  // needed; the halves are merged in the epilogue.
  static constexpr bool kHalfAcc = (D == 64) || !TANGENT;
  static constexpr uint32_t ACC_STRIDE = kHalfAcc ? 128 : 0;  // warpgroup w: TM_A + w * stride
  static constexpr uint32_t TM_A = 256;
  static constexpr uint32_t TM_T = 256 + D;
  static constexpr uint32_t TM_COLS = 512;
  static_assert(D == 64 || D == 128, "tensor-core path handles D = 64 or 128");
  static_assert(USED + 1024 <= 227 * 1024, "shared memory budget");
  static_assert(OFF_MSK % 1024 == 0, "the mask tile's 128-byte swizzle needs 1024-byte alignment");
};

constexpr int kSoftmaxThreads = 256;           // two warpgroups (warps 2..9)
// + producer warp (0), score-MMA warp (1) and P~V-MMA warp (10)
constexpr int kTcThreads = 96 + kSoftmaxThreads;
constexpr int kPvWarp = 10;
// Second score and P~V issuing warps (forward without tangents at D = 64,
// where a tile's products are narrow and one thread's issue rate paces them).
constexpr int kScoreWarp2 = 11, kPvWarp2 = 12;

// Control block in shared memory.
template <int NS>
struct TcCtrl {
  uint64_t q_full;
  uint64_t kdk_full[NS], kdk_empty[NS];
  uint64_t vdv_full[NS], vdv_empty[NS];
  // per score buffer (up to four); max_ready and xmax alternate by tile parity
  uint64_t s_full[4], p_full[4], max_ready[2];
  uint64_t s_ready[4];  // S of a score buffer is final (its dS may still be accumulating)
  uint64_t p_ready[4];  // P~ of a score buffer is stored (P~ * dS may not be yet)
  uint64_t o_full, drain, drain_pv, sums_ready;
  uint64_t drain2, drain_pv2;  // the second issuing threads' drains (split issue)
  uint64_t o_staged;  // every softmax warp has staged its O / tO rows in shared memory
  uint64_t pv_done[4];  // P~V MMAs of the tile in each score buffer are complete
  uint64_t ring_free, peer_ready;  // cluster split (arrived on by the other CTA)
  uint32_t tmem_base;
  int abort;
  float xmax[2][2][kTcBlockM];     // [tile parity][warpgroup][row] half-row maxima
  float xsum[2][4][kTcBlockM];     // [warpgroup][l, lx, mu, m][row] final half sums
  uint64_t dk_empty;               // the shared dK slot has been read (MTILE with tangents)
  uint64_t msk_full[2], msk_empty[2];  // the additive-mask slots in shared memory (MTILE)
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ void record_timeout(unsigned int* status, volatile int* abort) {
  *abort = 1;
  atomicOr(status, 1u);
}

// Bounded wait taken by every lane of a warp, with a warp-uniform outcome, so
// that the warp-collective TMEM instructions after it never run diverged.
// (Waiters sleep inside try_wait, so polling adds little shared-memory traffic.)
template <bool kHint = true>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* status,
                                          volatile int* abort) {
  const bool got = mbar_wait<kHint>(bar, parity, abort);
  if (!got) record_timeout(status, abort);
  return __all_sync(0xffffffffu, got);
}

// warp_wait for a barrier that another CTA of the cluster arrives on.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  unsigned int* status, volatile int* abort) {
  const bool got = mbar_wait_cluster(bar, parity, abort);
  if (!got) record_timeout(status, abort);
  return __all_sync(0xffffffffu, got);
}

// Loads the mask entries of one row for the KN keys starting at j0; entries at
// or beyond Nk are not read.  Bool masks pack 4 bytes per word.
template <int MASK, int KN>
struct MaskRegs {  // no per-row mask data for none / causal
  __device__ __forceinline__ void load(const FwdParams&, const void*, int) {}
};
template <int KN>
struct MaskRegs<kMaskBool, KN> {
  uint32_t w[KN / 4] = {};
  __device__ __forceinline__ void load(const FwdParams& p, const void* rowp, int j0) {
    const uint8_t* row = static_cast<const uint8_t*>(rowp);
    if (p.mask_vec && j0 + KN <= p.Nk) {
      const uint4* src = reinterpret_cast<const uint4*>(row + j0);
#pragma unroll
      for (int c = 0; c < KN / 16; ++c) {
        const uint4 x = __ldg(src + c);
        w[4 * c] = x.x; w[4 * c + 1] = x.y; w[4 * c + 2] = x.z; w[4 * c + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < KN / 4; ++c) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = j0 + 4 * c + e;
          const uint32_t byte = (j < p.Nk) ? row[static_cast<long long>(j) * p.msk] : 0u;
          word |= (byte != 0 ? 1u : 0u) << (8 * e);
        }
        w[c] = word;
      }
    }
  }
  __device__ __forceinline__ bool keep(int jj) const {
    return ((w[jj >> 2] >> (8 * (jj & 3))) & 0xFFu) != 0;
  }
};
template <int KN>
struct MaskRegs<kMaskAdditive, KN> {
  float a[KN] = {};
  __device__ __forceinline__ void load(const FwdParams& p, const void* rowp, int j0) {
    const float* row = static_cast<const float*>(rowp);
    if (p.mask_vec && j0 + KN <= p.Nk) {
      const float4* src = reinterpret_cast<const float4*>(row + j0);
#pragma unroll
      for (int c = 0; c < KN / 4; ++c) {
        const float4 x = __ldg(src + c);
        a[4 * c] = x.x; a[4 * c + 1] = x.y; a[4 * c + 2] = x.z; a[4 * c + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < KN; ++jj) {
        const int j = j0 + jj;
        a[jj] = (j < p.Nk) ? row[static_cast<long long>(j) * p.msk] : 0.0f;
      }
    }
  }
};

// Writes NP 16-byte pieces (8 16-bit values each) of row r, from column col
// on, into a [128 x D] tile in shared memory laid out as the TMA box of the
// output tensor map: 64-column chunks of 128 rows x 128 bytes, the 16-byte
// piece k of a row at position k ^ (row % 8) (128-byte swizzle).
// (tile_bytes and status serve the debug build's bounds check only.)
template <int NP>
__device__ __forceinline__ void stage_row(uint32_t tile, int r, int col,
                                          const uint32_t (&v)[NP * 4], uint32_t tile_bytes,
                                          unsigned int* status) {
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int cc = col + 8 * q;
    const uint32_t off = static_cast<uint32_t>((cc >> 6) * (kTcBlockM * 128) + r * 128 +
                                               ((((cc & 63) >> 3) ^ (r & 7)) << 4));
    if (JVP_CHECK(off + 16 <= tile_bytes && r < kTcBlockM, status, kChkSmem))
      st_shared_v4(tile + off, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

// Maximum of n values by a tree of three-input maxima (32 values: 17
// instructions, 4 dependent steps).
template <int N>
__device__ __forceinline__ float tree_max(const float (&x)[N]) {
  if constexpr (N == 1) {
    return x[0];
  } else if constexpr (N == 2) {
    return fmaxf(x[0], x[1]);
  } else {
    constexpr int M = (N + 2) / 3;
    float y[M];
#pragma unroll
    for (int k = 0; k < N / 3; ++k) y[k] = fmax3(x[3 * k], x[3 * k + 1], x[3 * k + 2]);
    if constexpr (N % 3 == 1) y[M - 1] = x[N - 1];
    if constexpr (N % 3 == 2) y[M - 1] = fmaxf(x[N - 2], x[N - 1]);
    return tree_max<M>(y);
  }
}

// One TMEM row piece of 32 or 64 columns of this thread's lane, into or out
// of registers (one wait for the load).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 32 || N == 64, "32 or 64 columns");
  if constexpr (N == 32) {
    tmem_ld32(taddr, r);
  } else {
    tmem_ld32x2(taddr, taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[0]),
                *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  }
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 16) {
    tmem_st16(taddr, r);
  } else {
    tmem_st32(taddr, r);
  }
}

// SPLIT: 0 single pass; kSplitWorkspace: split-KV over p.splits CTAs per
// query tile, partial states to p.split_ws for fwd_combine_kernel;
// kSplitCluster (D = 64): the key range of a query tile split between the two
// CTAs of a cluster, rank 1 handing its partial state to rank 0 through
// distributed shared memory.  The single-pass variant compiles without either.
constexpr int kSplitWorkspace = 1, kSplitCluster = 2;

// Receive area of the cluster split in rank 0 (inside its idle key/value
// rings, after the 2 x 16 KB where O and tO are staged): a float4
// {m, l, lx, mu~} per row, then one block per softmax warpgroup w holding,
// for each row, the fp32 A and T columns [32 w, 32 w + 32) of the peer (rows
// 16 bytes apart beyond their 64 floats, to spread shared-memory banks).  A
// softmax warp's 32 rows of a block are contiguous, so each warp sends its
// own part as soon as it has staged it.
constexpr int kPairRecvOffset = 32768;
constexpr int kPairRecvStats = 128 * 16;
constexpr int kPairRecvRowBytes = 2 * 32 * 4 + 16;
constexpr int kPairRecvBlock = 128 * kPairRecvRowBytes;
constexpr int kPairRecvBytes = kPairRecvStats + 2 * kPairRecvBlock;

// Whether the kernel brings the additive mask's tiles through a shared-memory
// slot (the layout parameter MTILE; kernel and launcher must agree).
template <int D, int MASK, bool TANGENT>
constexpr bool tc_mask_tile() {
  return MASK == kMaskAdditive && D == 128;
}
// Whether alternate tiles' products are issued by two score and two P~V
// threads (without tangents at D = 64, where whole tiles alternate between
// the warpgroups, so each accumulator still has one issuing thread), and the
// block size that follows.  Not with a mask: the two extra warps leave the
// boolean mask's two tiles of entries ahead too few registers.
template <int D, int MASK, bool TANGENT>
constexpr bool tc_split_issue() {
  return !TANGENT && D == 64 && (MASK == kMaskNone || MASK == kMaskCausal);
}
// Whether a second score warp issues the odd tiles' score products: with
// split issue above, and with tangents at D = 128 without a mask or causal
// (sixteen products per tile, eight of them N = 64, pace one issuing thread:
// bf16 B=4 H=16 N=2048 290.8 -> 280.9 us, causal 175.0 -> 172.2; with a
// boolean mask 301.6 -> 304.1 and at D = 64 202.0 -> 203.4, so not there).
// Each tile's products come from one thread, so their accumulation order
// stays fixed.
template <int D, int MASK, bool TANGENT, int SPLIT>
constexpr bool tc_score2() {
  return tc_split_issue<D, MASK, TANGENT>() ||
         (TANGENT && D == 128 && (MASK == kMaskNone || MASK == kMaskCausal) &&
          SPLIT != kSplitCluster);
}
template <int D, int MASK, bool TANGENT, int SPLIT>
constexpr int tc_threads() {
  return kTcThreads + (tc_score2<D, MASK, TANGENT, SPLIT>() ? 32 : 0) +
         (tc_split_issue<D, MASK, TANGENT>() ? 32 : 0);
}

template <typename T, int D, int MASK, bool TANGENT, int SPLIT>
__global__ void __launch_bounds__(tc_threads<D, MASK, TANGENT, SPLIT>(), 1)
    fwd_dual_tc_kernel(const __grid_constant__ TcMaps maps, const FwdParams p) {
  // The additive mask at D = 128 comes through shared memory when its layout
  // allows a tensor map (p.mask_tma), else by per-row loads in its tile (one
  // slot with tangents, two without).  (At D = 64 the registers hold a tile
  // ahead; the shared-memory slot measured slower there: its refill waits for
  // the previous tile's maximum and holds up the producer's deeper K/V rings.)
  constexpr bool kMTile = tc_mask_tile<D, MASK, TANGENT>();
  // Waits without a suspend-time hint at D = 64 (measured faster there).
  constexpr bool kHint = (D != 64);
  using L = TcLayout<D, TANGENT, kMTile>;
  constexpr int NMS = L::NMS > 0 ? L::NMS : 1;  // additive-mask slots (MTILE)
  constexpr bool kWsSplit = SPLIT == kSplitWorkspace;
  constexpr bool kPair = SPLIT == kSplitCluster;
  static_assert(!kPair || (D == 64 && TANGENT), "the cluster split is built for D = 64 with tangents");
  static_assert(!kPair || kPairRecvOffset + kPairRecvBytes <= L::OFF_CTRL - L::OFF_KDK,
                "cluster receive area fits the rings");
  constexpr int NS = L::NS;
  constexpr int BN = L::BN;
  constexpr int HN = BN / 2;  // key columns per softmax warpgroup
  // Without tangents at D = 128 the score products of two key tiles are
  // issued as one N = 128 product (see the score warp); not with a boolean
  // mask, where single tiles measured faster (bf16 B=4 H=16 N=2048: 187.5 us
  // against 190.3 with pairs taken by alternate warpgroups, 195.2 with the
  // pairs' ownership below), nor with an additive one (the same time either
  // way; its three-stage rings make room for two mask slots).
  constexpr bool kPairS = !TANGENT && D == 128 && (MASK == kMaskNone || MASK == kMaskCausal);
  // Without tangents (and without an additive mask) the two softmax
  // warpgroups take whole key tiles, each into its own accumulator, instead
  // of half of every tile: a thread's fixed per-tile costs (waits, TMEM round
  // trips, the row maximum, publishing) then cover 64 keys instead of 32.
  // Warpgroup w takes the tiles t with t % 2 == w, or, where the score
  // products come in pairs, the pairs with (t / 2) % 2 == w: the two tiles of
  // a pair complete together, so the warpgroups start their pairs one pair
  // apart rather than both at once (the warps of a sub-partition then do not
  // all want the exponential unit at the same time).
  constexpr bool kAlt = !TANGENT && MASK != kMaskAdditive;
  constexpr bool kPairOwn = kAlt && kPairS;
  constexpr bool kIssue2 = tc_split_issue<D, MASK, TANGENT>();  // second P~V warp
  constexpr bool kScore2 = tc_score2<D, MASK, TANGENT, SPLIT>();  // second score warp
  static_assert(!kIssue2 || (kAlt && !kPairS), "split issue: alternate single tiles");
  static_assert(!kScore2 || !kPairS, "a second score warp takes single tiles");
  constexpr int KW = kAlt ? BN : HN;  // keys of a tile per softmax thread
  // The next tile of the warpgroup that takes tile t, and whether tile t is
  // the first of its accumulator.
  auto next_tile = [](int t) {
    return kPairOwn ? t + ((t & 1) ? 3 : 1) : kAlt ? t + 2 : t + 1;
  };
  auto first_of_acc = [](int t) {
    return kPairOwn ? (t < 4 && (t & 1) == 0) : kAlt ? t < 2 : t == 0;
  };
  constexpr bool kBF16 = ElemTraits<T>::kBF16;
  constexpr int KSTEPS_D = D / 16;   // MMA K-steps over the head dimension
  constexpr int KSTEPS_N = BN / 16;  // MMA K-steps over a key tile
  constexpr int ACC_COLS = TANGENT ? 2 * D : D;  // TMEM columns of [A | T]
  constexpr uint32_t IDESC_S = idesc_f16(kBF16, 128, TANGENT ? 2 * BN : BN, false);
  constexpr uint32_t IDESC_S2 = idesc_f16(kBF16, 128, 2 * BN, false);  // S of two key tiles
  constexpr uint32_t IDESC_DS = idesc_f16(kBF16, 128, BN, false);
  constexpr uint32_t IDESC_AT = idesc_f16(kBF16, 128, ACC_COLS, true);
  constexpr uint32_t IDESC_T = idesc_f16(kBF16, 128, D, true);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle pattern.
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  static_assert(sizeof(TcCtrl<NS>) <= L::CTRL_BYTES, "control block budget");
  TcCtrl<NS>* ctrl = reinterpret_cast<TcCtrl<NS>*>(smem + L::OFF_CTRL);
  volatile int* abort = &ctrl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: heads are taken in groups sized to about one wave of CTAs,
  // with the query tiles of a group innermost, so that the K/V of the heads in
  // flight stay in L2.  Causal problems take their longest tiles first.
  const int BH = p.B * p.H;
  const int nq = p.num_q_tiles;
  const int G = p.group_heads;
  // Split-KV: the p.splits CTAs of one (query tile, head) are adjacent.
  const int split = SPLIT ? static_cast<int>(blockIdx.x % p.splits) : 0;
  const int item = SPLIT ? static_cast<int>(blockIdx.x / p.splits) : static_cast<int>(blockIdx.x);
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
  const int q0 = qt * L::BM;
  int n_kv = (p.Nk + BN - 1) / BN;
  if (causal) {
    const int last_row = min(q0 + L::BM, p.Nq) - 1;
    n_kv = min(n_kv, last_row / BN + 1);
  }
  // This CTA's key tiles: [kv0, kv0 + n_kv) (the whole range unless split).
  int kv0 = 0;
  if constexpr (SPLIT) {
    const int per_split = (n_kv + p.splits - 1) / p.splits;
    kv0 = min(n_kv, split * per_split);
    n_kv = min(n_kv, kv0 + per_split) - kv0;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctrl->kdk_full[s], 1);
      mbar_init(&ctrl->kdk_empty[s], 1);
      mbar_init(&ctrl->vdv_full[s], 1);
      mbar_init(&ctrl->vdv_empty[s], 1);
    }
    for (int s = 0; s < L::NB; ++s) {
      mbar_init(&ctrl->s_full[s], 1);
      mbar_init(&ctrl->s_ready[s], 1);
      mbar_init(&ctrl->p_ready[s], kSoftmaxThreads / 32);
      // one arrival per softmax warp working on the buffer's tile
      mbar_init(&ctrl->p_full[s], (kAlt ? kSoftmaxThreads / 2 : kSoftmaxThreads) / 32);
      mbar_init(&ctrl->pv_done[s], 1);
    }
    mbar_init(&ctrl->max_ready[0], kSoftmaxThreads / 32);
    mbar_init(&ctrl->max_ready[1], kSoftmaxThreads / 32);
    mbar_init(&ctrl->drain_pv, 1);
    mbar_init(&ctrl->o_full, kIssue2 ? 2 : 1);  // one commit per P~V-issuing thread
    mbar_init(&ctrl->drain, 1);
    mbar_init(&ctrl->drain2, 1);
    mbar_init(&ctrl->drain_pv2, 1);
    mbar_init(&ctrl->sums_ready, kSoftmaxThreads);
    mbar_init(&ctrl->o_staged, kSoftmaxThreads / 32);
    mbar_init(&ctrl->ring_free, 1);    // cluster split: rank 0's rings are idle
    mbar_init(&ctrl->peer_ready, 1);   // cluster split: rank 1's state has landed (with bytes)
    mbar_init(&ctrl->dk_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->msk_full[s], 1);
      mbar_init(&ctrl->msk_empty[s], kSoftmaxThreads / 32);
    }
    ctrl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, L::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // Cluster split: every thread arrives once its CTA's barriers are
  // initialised; a thread that touches the other CTA waits for the cluster
  // first (the rest wait before exiting).
  if constexpr (kPair) cluster_arrive();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      if (TANGENT) {
        tma_prefetch_desc(&maps.dq);
        tma_prefetch_desc(&maps.dk);
        tma_prefetch_desc(&maps.dv);
      }
      const bool mtma = kMTile && p.mask_tma;
      // mask coordinates: a broadcast dimension of the mask has extent 1
      const int mh = p.msh ? h : 0, mb = p.msb ? b : 0;
      if (mtma) tma_prefetch_desc(&maps.msk);
      mbar_arrive_expect_tx(&ctrl->q_full, (TANGENT ? 2 : 1) * L::Q_BYTES);
      for (int c = 0; c < L::KCH; ++c) {
        tma_load_4d(smem + L::OFF_Q + c * L::BM * 128, &maps.q, &ctrl->q_full, c * 64, q0, h, b);
        if (TANGENT)
          tma_load_4d(smem + L::OFF_DQ + c * L::BM * 128, &maps.dq, &ctrl->q_full, c * 64, q0, h,
                      b);
      }
      int k_fills = 0, v_fills = 0, m_fills = 0;  // ring fills issued so far
      // Key tile u into stage u % NS once the stage's previous score products
      // are done.  The K tiles are issued KLEAD tiles ahead
      // of the V tiles (whose stages wait for the far later P~V products), so
      // both tiles of a score pair have landed when the pair's buffers free
      // (with paired score products).
      constexpr int KLEAD = kPairS ? 2 : 0;
      auto load_k = [&](int u) -> bool {
        const int su = u % NS;
        if (!mbar_wait<kHint>(&ctrl->kdk_empty[su], ((u / NS) & 1) ^ 1, abort) ||
            (L::kSharedDK && !mbar_wait<kHint>(&ctrl->dk_empty, (u & 1) ^ 1, abort)))
          return false;
        const int ju = (kv0 + u) * BN;
        mbar_arrive_expect_tx(&ctrl->kdk_full[su], L::KDK_BYTES);
        for (int c = 0; c < L::KCH; ++c) {
          tma_load_4d(smem + L::k_off(su, c), &maps.k, &ctrl->kdk_full[su], c * 64, ju, hk, b);
          if (TANGENT)
            tma_load_4d(smem + L::dk_off(su, c), &maps.dk, &ctrl->kdk_full[su], c * 64, ju, hk,
                        b);
        }
        ++k_fills;
        return true;
      };
      bool k_ok = true;
      for (int u = 0; k_ok && u < KLEAD && u < n_kv; ++u) k_ok = load_k(u);
      if (!k_ok) record_timeout(p.status, abort);
      for (int t = 0; k_ok && t < n_kv; ++t) {
        const int s = t % NS;
        const uint32_t ph = (t / NS) & 1;
        const int j0 = (kv0 + t) * BN;
        if (t + KLEAD < n_kv && !load_k(t + KLEAD)) {
          record_timeout(p.status, abort);
          break;
        }
        if (mtma) {
          // slot t % NMS: tile t's mask once every softmax warp has read the
          // slot's previous tile (t - NMS)
          const int ms = t % NMS;
          if (!mbar_wait<kHint>(&ctrl->msk_empty[ms], ((t / NMS) & 1) ^ 1, abort)) {
            record_timeout(p.status, abort);
            break;
          }
          mbar_arrive_expect_tx(&ctrl->msk_full[ms], L::MSK_TILE);
          for (int w = 0; w < 2; ++w)
            tma_load_4d(smem + L::OFF_MSK + ms * L::MSK_TILE + w * L::BM * 128, &maps.msk,
                        &ctrl->msk_full[ms], j0 + w * (BN / 2), q0, mh, mb);
          ++m_fills;
        }
        if (!mbar_wait<kHint>(&ctrl->vdv_empty[s], ph ^ 1, abort)) {
          record_timeout(p.status, abort);
          break;
        }
        uint8_t* vdv = smem + L::OFF_VDV + s * L::VDV_BYTES;
        mbar_arrive_expect_tx(&ctrl->vdv_full[s], L::VDV_BYTES);
        for (int c = 0; c < L::KCH; ++c) {
          tma_load_4d(vdv + c * L::VCHUNK_BYTES, &maps.v, &ctrl->vdv_full[s], c * 64, j0, hk, b);
          if (TANGENT)
            tma_load_4d(vdv + (L::KCH + c) * L::VCHUNK_BYTES, &maps.dv, &ctrl->vdv_full[s], c * 64,
                        j0, hk, b);
        }
        ++v_fills;
      }
      if (*abort) {
        // Let every copy already issued land before the CTA can exit.
        const int zero = 0;
        mbar_wait<kHint>(&ctrl->q_full, 0, &zero);
        for (int t = max(0, k_fills - NS); t < k_fills; ++t)
          mbar_wait<kHint>(&ctrl->kdk_full[t % NS], (t / NS) & 1, &zero);
        for (int t = max(0, v_fills - NS); t < v_fills; ++t)
          mbar_wait<kHint>(&ctrl->vdv_full[t % NS], (t / NS) & 1, &zero);
        for (int u = max(0, m_fills - NMS); u < m_fills; ++u)
          mbar_wait<kHint>(&ctrl->msk_full[u % NMS], (u / NMS) & 1, &zero);
      }
    }
  } else if (warp == 1 || (kScore2 && warp == kScoreWarp2)) {
    // ------------------------------------------------------------ score MMAs
    // Tile t's score products go into buffer t % NB once its K tile has landed
    // and the P~V MMAs of tile t - NB (the buffer's previous user) are done.
    // Two issuing threads (this one and the P~V warp) keep the tensor pipe fed
    // while either waits, and interleave the narrow dQ K^T products.  Without
    // tangents at D = 128 the products of two key tiles (t even, t + 1) are issued as
    // one pair of N = 128 products into the adjacent buffers t % 4 and
    // t % 4 + 1 from the adjacent stages t % 4 and t % 4 + 1: half the
    // instructions of two N = 64 sets (one thread issues a tcgen05.mma about
    // every 70 cycles) and less tensor time (a narrow product is paced by
    // reading its A tile from shared memory).  With split issue this warp
    // takes the even tiles and the second score warp the odd ones.
    static_assert(!kPairS || (NS % 2 == 0 && L::NB % 2 == 0), "pairs of stages and buffers");
    if (lane == 0) {
      bool ok = mbar_wait<kHint>(&ctrl->q_full, 0, abort);
      tc_fence_after();
      const uint32_t sQ = smem_u32(smem + L::OFF_Q);
      const uint32_t sdQ = smem_u32(smem + L::OFF_DQ);
      // s < 0: -Q K^T, -Q dK^T, -dQ K^T (negate-A bit), with |s| applied later.
      const uint32_t neg_a = p.neg_scores ? (1u << 13) : 0u;
      constexpr int SSTEP = (kPairS || kScore2) ? 2 : 1;  // key tiles per step
      const int s_first = (kScore2 && warp != 1) ? 1 : 0;
      uint64_t* const s_drain = (kScore2 && warp != 1) ? &ctrl->drain2 : &ctrl->drain;
      for (int t = s_first; ok && t < n_kv; t += SSTEP) {
        const bool pair = kPairS && t + 1 < n_kv;
        const int s = t % NS;
        const int bb = t % L::NB;  // score buffer
        if (t >= L::NB && !mbar_wait<kHint>(&ctrl->pv_done[bb], ((t - L::NB) / L::NB) & 1, abort)) {
          ok = false;
          break;
        }
        if (pair && t + 1 >= L::NB &&
            !mbar_wait<kHint>(&ctrl->pv_done[bb + 1], ((t + 1 - L::NB) / L::NB) & 1, abort)) {
          ok = false;
          break;
        }
        if (!mbar_wait<kHint>(&ctrl->kdk_full[s], (t / NS) & 1, abort) ||
            (pair && !mbar_wait<kHint>(&ctrl->kdk_full[s + 1], ((t + 1) / NS) & 1, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // stage s: chunk c of the first product's operand at sM + c * kChunk,
        // of the K rows at sK + c * kChunk
        const uint32_t sK = smem_u32(smem + L::k_off(s, 0));
        const uint32_t sM = smem_u32(smem + L::m1_off(s, 0));
        constexpr int kChunk = L::K_CHUNK_STRIDE;
        const uint32_t d_s = tmem + L::buf_col(bb);
#pragma unroll
        for (int kk = 0; kk < KSTEPS_D; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sQ + (kk >> 2) * L::BM * 128 + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(sM + (kk >> 2) * kChunk + off, 16, 1024);
          mma_ss(d_s, a, bd, (pair ? IDESC_S2 : IDESC_S) | neg_a, kk > 0 ? 1u : 0u);
        }
        // S is complete: the softmax starts on it while dQ K^T accumulates into dS.
        if (TANGENT) mma_commit(&ctrl->s_ready[bb]);
        if (L::kSharedDK) mma_commit(&ctrl->dk_empty);  // dK is read only by that product
        if (TANGENT) {
#pragma unroll
          for (int kk = 0; kk < KSTEPS_D; ++kk) {
            const uint32_t off = (kk & 3) * 32;
            const uint64_t a = sdesc_sw128(sdQ + (kk >> 2) * L::BM * 128 + off, 16, 1024);
            const uint64_t bd = sdesc_sw128(sK + (kk >> 2) * kChunk + off, 16, 1024);
            mma_ss(tmem + L::ds_col(bb), a, bd, IDESC_DS | neg_a, 1u);
          }
        }
        mma_commit(&ctrl->kdk_empty[s]);
        if (pair) mma_commit(&ctrl->kdk_empty[s + 1]);
        mma_commit(&ctrl->s_full[bb]);
        if (pair) mma_commit(&ctrl->s_full[bb + 1]);
      }
      if (!ok) record_timeout(p.status, abort);
      // Drain: every MMA this thread issued completes before TMEM is freed.
      mma_commit(s_drain);
      const int zero = 0;
      mbar_wait<kHint>(s_drain, 0, &zero);
    }
  } else if (warp == kPvWarp || (kIssue2 && warp == kPvWarp2)) {
    // ------------------------------------------------------------ P~V MMAs
    // (with split issue: this warp the even tiles, the second P~V warp the odd
    // ones, each into its warpgroup's accumulator)
    if (lane == 0) {
      bool ok = true;
      const int p_first = (kIssue2 && warp != kPvWarp) ? 1 : 0;
      uint64_t* const p_drain = (kIssue2 && warp != kPvWarp) ? &ctrl->drain_pv2 : &ctrl->drain_pv;
      for (int t = p_first; ok && t < n_kv; t += kIssue2 ? 2 : 1) {
        const int buf = t % L::NB;
        const uint32_t bph = (t / L::NB) & 1;
        if (!mbar_wait<kHint>(TANGENT ? &ctrl->p_ready[buf] : &ctrl->p_full[buf], bph, abort)) {
          ok = false;
          break;
        }
        const int s = t % NS;
        if (!mbar_wait<kHint>(&ctrl->vdv_full[s], (t / NS) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + L::OFF_VDV + s * L::VDV_BYTES);
        // P~ (16-bit pairs) of keys [16 kk, 16 kk + 16): with per-warpgroup
        // accumulators warpgroup kk / 2 stored them at the start of its own S
        // columns, otherwise they are packed; P~ * dS, BN columns further, is
        // always at the start of the warpgroup's own dS columns.
        const uint32_t p_tm = tmem + L::s_col(buf);
        const uint32_t pd_tm = tmem + L::ds_col(buf);
        auto pcol = [](int kk) -> uint32_t {
          return (L::kHalfAcc && !kAlt)
                     ? static_cast<uint32_t>((kk / (HN / 16)) * HN + (kk % (HN / 16)) * 8)
                     : static_cast<uint32_t>(kk * 8);
        };
        // P~ * dS always sits at the start of its warpgroup's own dS columns.
        auto pdcol = [](int kk) -> uint32_t {
          return static_cast<uint32_t>((kk / (HN / 16)) * HN + (kk % (HN / 16)) * 8);
        };
        // With per-warpgroup accumulators, K-steps [w * KH, w * KH + KH) (the
        // keys of warpgroup w) go to warpgroup w's [A | T]; with whole tiles,
        // all of tile t's go to the accumulator of the warpgroup that took it.
        constexpr int KH = (L::kHalfAcc && !kAlt) ? KSTEPS_N / 2 : KSTEPS_N;
#pragma unroll
        for (int kk = 0; kk < KSTEPS_N; ++kk) {
          const uint64_t bd = sdesc_sw128(sV + kk * 16 * 128, L::VCHUNK_BYTES, 1024);
          const int acc_w = kPairOwn ? ((t >> 1) & 1) : kAlt ? (t & 1) : kk / KH;
          const uint32_t acc_base = tmem + L::TM_A + acc_w * L::ACC_STRIDE;
          mma_ts(acc_base, p_tm + pcol(kk), bd, IDESC_AT,
                 (!first_of_acc(t) || kk % KH > 0) ? 1u : 0u);
        }
        if (TANGENT) {
          if (!mbar_wait<kHint>(&ctrl->p_full[buf], bph, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < KSTEPS_N; ++kk) {
            const uint64_t bd = sdesc_sw128(sV + kk * 16 * 128, L::VCHUNK_BYTES, 1024);
            mma_ts(tmem + L::TM_T + (kk / KH) * L::ACC_STRIDE, pd_tm + pdcol(kk), bd, IDESC_T, 1u);
          }
        }
        mma_commit(&ctrl->vdv_empty[s]);
        mma_commit(&ctrl->pv_done[buf]);
      }
      if (ok) {
        mma_commit(&ctrl->o_full);
      } else {
        record_timeout(p.status, abort);
      }
      mma_commit(p_drain);
      const int zero = 0;
      mbar_wait<kHint>(p_drain, 0, &zero);
    }
  } else if (warp >= 2 && warp < 2 + kSoftmaxThreads / 32) {
    // ------------------------------------------------------------ softmax
    // Two warpgroups; warpgroup wg owns key columns [wg*HN, wg*HN + HN) of
    // every tile (with alternate tiles: every column of tiles wg, wg + 2, ...)
    // and, in the epilogue, output columns [wg*D/2, wg*D/2 + D/2).
    // Thread (warp, lane) owns query row r = 32 * (warp % 4) + lane (its TMEM lane).
    const int wg = (warp - 2) >> 2;
    const int sub = warp & 3;
    const int r = sub * 32 + lane;
    const int i = q0 + r;
    const bool row_ok = i < p.Nq;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const int cofs = kAlt ? 0 : wg * HN;
    const float c = p.scale_log2;
    const float s_scale = p.scale;
    float m_run = -INFINITY;  // running max, log2 units of the scaled logits (whole row)
    float l_run = 0.0f;       // this half's sum of p~ as rounded for the MMA
    float lx_run = 0.0f;      // this half's sum of p~ in fp32 (for the log-sum-exp)
    float mu_run = 0.0f;      // this half's sum of p~ * dS as rounded for the MMA
    bool ok = true;

    const void* mrow = nullptr;
    if (MASK == kMaskBool || MASK == kMaskAdditive) {
      const long long off = static_cast<long long>(b) * p.msb + static_cast<long long>(h) * p.msh +
                            static_cast<long long>(row_ok ? i : 0) * p.msq;
      mrow = (MASK == kMaskBool)
                 ? static_cast<const void*>(static_cast<const uint8_t*>(p.mask) + off)
                 : static_cast<const void*>(static_cast<const float*>(p.mask) + off);
    }

    // Mask entries are loaded one tile ahead, so their global-memory latency
    // overlaps a whole tile of work (not the additive mask at D = 128, whose
    // two tiles of 32 floats would not fit the register budget next to the
    // tangent terms, and which comes through shared memory).
    constexpr bool kMaskAhead = !tc_mask_tile<D, MASK, TANGENT>();
    const bool mstaged = kMTile && p.mask_tma;  // additive tiles through shared memory (D = 128)
    const int t_first = kPairOwn ? 2 * wg : kAlt ? wg : 0;
    // The next own tile's entries (with whole tiles also the one after it:
    // with paired ownership the next tile may follow at once).
    MaskRegs<MASK, KW> mnext, mnext2;
    if (kMaskAhead && !mstaged && row_ok && t_first < n_kv) {
      mnext.load(p, mrow, (kv0 + t_first) * BN + cofs);
      if (kAlt && next_tile(t_first) < n_kv)
        mnext2.load(p, mrow, (kv0 + next_tile(t_first)) * BN + cofs);
    }
    for (int t = t_first; t < n_kv; t = next_tile(t)) {
      const int buf = t % L::NB;  // score buffer
      const uint32_t bph = (t / L::NB) & 1;
      const int xb = t & 1;       // tile parity: the maxima exchange slot
      const int j0 = (kv0 + t) * BN + cofs;  // first key of this thread's part of the tile
      MaskRegs<MASK, KW> mreg;
      if constexpr (kMTile) {
        if (mstaged) {
          // The tile's entries were copied into shared memory by TMA a tile
          // ahead, one [128 x 32] box per warpgroup with the 128-byte
          // swizzle: 16-byte piece c of row r sits at piece position
          // c ^ (r % 8), so the 8 rows of a quarter warp hit distinct banks.
          // (The slot is released once the entries are consumed, below.)
          if (!warp_wait<kHint>(&ctrl->msk_full[t % NMS], (t / NMS) & 1, p.status, abort)) {
            ok = false;
            break;
          }
          const uint32_t mrow_s = smem_u32(smem + L::OFF_MSK + (t % NMS) * L::MSK_TILE +
                                           wg * L::BM * 128 + r * 128);
#pragma unroll
          for (int c4 = 0; c4 < HN / 4; ++c4) {
            const float4 v = ld_shared_v4f(mrow_s + ((c4 ^ (r & 7)) << 4));
            mreg.a[4 * c4] = v.x;
            mreg.a[4 * c4 + 1] = v.y;
            mreg.a[4 * c4 + 2] = v.z;
            mreg.a[4 * c4 + 3] = v.w;
          }
        }
      }
      if (!mstaged) {
        if constexpr (kMaskAhead) {
          mreg = mnext;
          if constexpr (kAlt) {
            mnext = mnext2;
            const int t2 = next_tile(next_tile(t));
            if (row_ok && t2 < n_kv) mnext2.load(p, mrow, (kv0 + t2) * BN + cofs);
          } else {
            if (row_ok && t + 1 < n_kv) mnext.load(p, mrow, j0 + BN);
          }
          if constexpr (MASK == kMaskAdditive) {
            // additive entries two tiles ahead into L2 as well (measured: bool
            // masks, a quarter the bytes, do not gain)
            if (row_ok && p.msk == 1 && t + 2 < n_kv && j0 + 2 * BN < p.Nk)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const float*>(mrow) + j0 +
                                                            2 * BN));
          }
        } else if (row_ok) {
          // The next two tiles' entries of this row (one 128-byte line each for
          // contiguous keys) are prefetched into L2, so those in-tile loads hit
          // there (no registers to hold them a tile ahead at D = 128).
          if (p.msk == 1) {
            const float* rowf = static_cast<const float*>(mrow);
            if (t + 1 < n_kv && j0 + BN < p.Nk)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(rowf + j0 + BN));
            if (t + 2 < n_kv && j0 + 2 * BN < p.Nk)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(rowf + j0 + 2 * BN));
          }
          mreg.load(p, mrow, j0);
        }
      }
      // With tangents, S is read as soon as it is final and dS (whose
      // dQ K^T part is still accumulating) only when the tangent terms need it.
      if (!warp_wait<kHint>(TANGENT ? &ctrl->s_ready[buf] : &ctrl->s_full[buf], bph, p.status,
                     abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sa[KW], da[HN];  // S and dS (raw, unscaled) of this thread's keys
      if (JVP_CHECK(L::s_col(buf) + cofs + KW <= L::TM_COLS, p.status, kChkTmem))
        tmem_ld_cols(lane_base + L::s_col(buf) + cofs, sa);
      float x[KW];
#pragma unroll
      for (int jj = 0; jj < KW; ++jj) x[jj] = __uint_as_float(sa[jj]);
      // Masking (raw-score domain unless additive, which is pre-scaled).
      if constexpr (MASK == kMaskAdditive) {
#pragma unroll
        for (int jj = 0; jj < HN; ++jj) x[jj] = fmaf(x[jj], c, mreg.a[jj] * kLog2e);
      } else if constexpr (MASK == kMaskBool) {
#pragma unroll
        for (int jj = 0; jj < KW; ++jj)
          if (!mreg.keep(jj)) x[jj] = -INFINITY;
      }
      if (j0 + KW > p.Nk) {
#pragma unroll
        for (int jj = 0; jj < KW; ++jj)
          if (j0 + jj >= p.Nk) x[jj] = -INFINITY;
      }
      if (causal && j0 + KW - 1 > q0) {
#pragma unroll
        for (int jj = 0; jj < KW; ++jj)
          if (j0 + jj > i) x[jj] = -INFINITY;
      }
      // p~ = 2^(x - m_use) (kept in e), P~ packed to 16 bits, and the sums of
      // the packed values (l) and of the fp32 p~ (lx); x is left as it is.
      uint32_t pk[KW / 2], pdk[HN / 2];
      float e[KW];
      float l_part = 0.f, lx_part = 0.f, mu_part = 0.f;
      auto weights = [&](float m_use) {
        if (MASK == kMaskAdditive) {
#pragma unroll
          for (int jj = 0; jj < KW; ++jj) e[jj] = ex2_approx(x[jj] - m_use);
        } else {
          const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_use, -m_use);
#pragma unroll
          for (int jj = 0; jj < KW; jj += 2) {
            const float2 arg = fma2(make_float2(x[jj], x[jj + 1]), c2, nm2);
            e[jj] = ex2_approx(arg.x);
            e[jj + 1] = ex2_approx(arg.y);
          }
        }
        float2 lsum[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        float2 xsum[2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int jj = 0; jj < KW; jj += 2) {
          pk[jj >> 1] = ElemTraits<T>::pack(e[jj], e[jj + 1]);
          lsum[(jj >> 1) & 3] = add2(lsum[(jj >> 1) & 3], ElemTraits<T>::unpack(pk[jj >> 1]));
          xsum[(jj >> 1) & 1] = add2(xsum[(jj >> 1) & 1], make_float2(e[jj], e[jj + 1]));
        }
        l_part = (lsum[0].x + lsum[0].y) + (lsum[1].x + lsum[1].y) + (lsum[2].x + lsum[2].y) +
                 (lsum[3].x + lsum[3].y);
        lx_part = (xsum[0].x + xsum[0].y) + (xsum[1].x + xsum[1].y);
      };
      // P~ * s * dS packed to 16 bits and the sum of the packed values (mu~).
      auto tangent_terms = [&]() {
        {
          float2 msum[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
          const float2 s2 = make_float2(s_scale, s_scale);
#pragma unroll
          for (int jj = 0; jj < HN; jj += 2) {
            const float2 ds = make_float2(__uint_as_float(da[jj]), __uint_as_float(da[jj + 1]));
            const float2 pd = mul2(make_float2(e[jj], e[jj + 1]), mul2(ds, s2));
            pdk[jj >> 1] = ElemTraits<T>::pack(pd.x, pd.y);
            msum[(jj >> 1) & 3] = add2(msum[(jj >> 1) & 3], ElemTraits<T>::unpack(pdk[jj >> 1]));
          }
          mu_part = (msum[0].x + msum[0].y) + (msum[1].x + msum[1].y) + (msum[2].x + msum[2].y) +
                    (msum[3].x + msum[3].y);
        }
      };
      const float mx = tree_max(x);
      const float m_half = (MASK == kMaskAdditive) ? mx : mx * c;
      float m_tile = m_half;
      bool spec = false;  // weights already computed with the unchanged row maximum
      if constexpr (!L::kHalfAcc) {
        // Exchange the half-row maxima between the two warpgroups.  Until the
        // other half's maximum is in, assume the row maximum stays (the usual
        // case after the first tile) and compute the weights with it; the
        // decision below is the same either way, so is every value stored.
        ctrl->xmax[xb][wg][r] = m_half;
        // A mask tile read from shared memory is consumed once m_half is
        // stored (it depends on every entry, so each lane's reads of the slot
        // have returned before that store issues): release the slot for the
        // next tile's copy, the reads ordered before the copy's writes.
        if (mstaged) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctrl->max_ready[xb]);
          if (mstaged) mbar_arrive(&ctrl->msk_empty[t % NMS]);
        }
        spec = __all_sync(0xffffffffu,
                          m_run != -INFINITY && !(m_half > m_run + kRescaleThreshold));
        if (spec) weights(m_run);
        if (!warp_wait<kHint>(&ctrl->max_ready[xb], (t >> 1) & 1, p.status, abort)) {
          ok = false;
          break;
        }
        m_tile = fmaxf(m_half, ctrl->xmax[xb][wg ^ 1][r]);
      } else if (mstaged) {
        // No exchange here: the same store of the half-row maximum (into the
        // otherwise unused exchange area) orders the mask slot's reads before
        // its release.
        ctrl->xmax[xb][wg][r] = m_half;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->msk_empty[t % NMS]);
      }
      const bool need = m_tile > m_run + kRescaleThreshold;
      if (!spec || __any_sync(0xffffffffu, need)) {
        const float m_new = need ? m_tile : m_run;
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
        l_run *= alpha;
        lx_run *= alpha;
        mu_run *= alpha;
        if (!first_of_acc(t) && __any_sync(0xffffffffu, need)) {
          // A and T hold tile t-1's contributions once its MMAs are done (with
          // whole tiles the accumulator's last tile may be t - 3; tile t - 1's
          // products complete after it); each warpgroup rescales half of the
          // [A | T] columns of its rows.  The wait is on the completions of
          // tile t - 1's score buffer, which a parity wait follows exactly:
          // the buffer's previous user, tile t - 1 - NB, is done (tile t's
          // scores needed tile t - NB's products done), and its next, tile
          // t - 1 + NB, cannot be before this thread publishes tile t's P~.
          // (One barrier for all tiles would not do: with four buffers its
          // completions may lag tile t - 1 by three, and a parity wait cannot
          // tell a phase from the one two before it.)
          // (With split issue the accumulator's products come from one thread
          // whose commits cover only its own: wait on its last tile, t - 2,
          // exact by the same argument with t - 2 for t - 1.)
          const int tb = kIssue2 ? t - 2 : t - 1;
          if (!warp_wait<kHint>(&ctrl->pv_done[tb % L::NB], (tb / L::NB) & 1, p.status, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Shared accumulator: each warpgroup rescales half of its columns;
          // per-warpgroup accumulators: each rescales its own.
          const int c_lo = L::kHalfAcc ? 0 : wg * (ACC_COLS / 2);
          const int c_hi = L::kHalfAcc ? ACC_COLS : (wg + 1) * (ACC_COLS / 2);
          const uint32_t a_base = lane_base + L::TM_A + wg * L::ACC_STRIDE;
#pragma unroll 1
          for (int col = c_lo; col < c_hi; col += 32) {
            uint32_t acc[32];
            if (!JVP_CHECK(L::TM_A + wg * L::ACC_STRIDE + col + 32 <= L::TM_COLS, p.status,
                           kChkTmem))
              continue;
            tmem_ld32(a_base + col, acc);
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = __float_as_uint(__uint_as_float(acc[e]) * alpha);
            tmem_st32(a_base + col, acc);
          }
          tmem_st_wait();
        }
        m_run = m_new;
        weights((m_run == -INFINITY) ? 0.0f : m_run);
      }
      l_run += l_part;
      lx_run += lx_part;
      // Where P~ goes: with per-warpgroup accumulators (no per-tile exchange)
      // into this warpgroup's own S columns, already read, since the other
      // warpgroup may still be reading its scores; otherwise the exchange has
      // ordered both warpgroups' reads first and the two halves are packed
      // side by side.
      const uint32_t pofs = L::kHalfAcc ? cofs : wg * (HN / 2);
      if (JVP_CHECK(L::s_col(buf) + pofs + KW / 2 <= L::TM_COLS, p.status, kChkTmem))
        tmem_st_cols(lane_base + L::s_col(buf) + pofs, pk);
      if (TANGENT) {
        // Publish P~ first: the P~ [V | dV] products run while the tangent
        // terms wait for dS.
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->p_ready[buf]);
        // dS is complete once the buffer's dQ K^T products are; P~ * dS goes
        // into this warpgroup's own dS columns (the other warpgroup may not
        // have read its dS yet).
        if (!warp_wait<kHint>(&ctrl->s_full[buf], bph, p.status, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (JVP_CHECK(L::ds_col(buf) + cofs + 32 <= L::TM_COLS, p.status, kChkTmem))
          tmem_ld32(lane_base + L::ds_col(buf) + cofs, da);
        tangent_terms();
        mu_run += mu_part;
        if (JVP_CHECK(L::ds_col(buf) + cofs + 16 <= L::TM_COLS, p.status, kChkTmem))
          tmem_st16(lane_base + L::ds_col(buf) + cofs, pdk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->p_full[buf]);  // one arrival per softmax warp
    }

    // ------------------------------------------------------------ epilogue
    // Combine the two halves' sums (both warpgroups hold the same m_run).
    if (ok) {
      ctrl->xsum[wg][0][r] = l_run;
      ctrl->xsum[wg][1][r] = lx_run;
      ctrl->xsum[wg][2][r] = mu_run;
      ctrl->xsum[wg][3][r] = m_run;
      mbar_arrive(&ctrl->sums_ready);
      ok = warp_wait<kHint>(&ctrl->sums_ready, 0, p.status, abort);
    }
    // The accumulators are final once the last P~V products are: the cluster
    // split waits here (rank 0's rings are then idle for the peer's state),
    // the other variants only before their first TMEM load, so the row
    // statistics below are formed while those products finish.
    if (kPair && ok && n_kv > 0) ok = warp_wait<kHint>(&ctrl->o_full, 0, p.status, abort);
    auto wait_acc = [&]() {
      if (!kPair && ok && n_kv > 0) ok = warp_wait<kHint>(&ctrl->o_full, 0, p.status, abort);
      tc_fence_after();
    };
    // O and tO rows are staged in the (now idle) [K;dK] ring, laid out as the
    // output tensor maps' 128-row boxes, and written by TMA stores: a warp
    // storing its own 32 rows directly would touch 32 lines per instruction.
    const uint32_t o_tile = smem_u32(smem + L::OFF_KDK);
    const uint32_t t_tile = o_tile + L::KCH * L::BM * 128;
    static_assert((TANGENT ? 2 : 1) * L::KCH * L::BM * 128 <= L::OFF_CTRL - L::OFF_KDK,
                  "output staging fits the key/value rings");
    if constexpr (kPair) {
      if (warp == 2) cluster_wait();  // both CTAs' barriers are initialised
      if (split == 0 && warp == 2 && lane == 0) {
        // the peer's state arrives as one bulk copy into the idle rings
        mbar_arrive_expect_tx(&ctrl->peer_ready, kPairRecvBytes);
        // Rank 0's rings are idle once its MMAs are done: rank 1 may fill them.
        if (ok) mbar_arrive_cluster(cluster_map(smem_u32(&ctrl->ring_free), 1));
      }
    }
    if (L::kHalfAcc && ok) {
      // Merge of the two warpgroups' states (each relative to its own max):
      // with M = max(m_0, m_1) and a_w = 2^(m_w - M), l = sum a_w l_w (so for
      // lx, mu~) and A = sum a_w A_w, T = sum a_w T_w, then the usual epilogue
      // (or, split-KV, the merged partial state; or, cluster split, the same
      // merge once more with the peer CTA's state).
      const float m_oth = ctrl->xsum[wg ^ 1][3][r];
      const float m_all = fmaxf(m_run, m_oth);
      const float a_own = (m_run == -INFINITY) ? 0.0f : exp2f(m_run - m_all);
      const float a_oth = (m_oth == -INFINITY) ? 0.0f : exp2f(m_oth - m_all);
      const float l_all = a_own * l_run + a_oth * ctrl->xsum[wg ^ 1][0][r];
      const float lx_all = a_own * lx_run + a_oth * ctrl->xsum[wg ^ 1][1][r];
      const float mu_all = a_own * mu_run + a_oth * ctrl->xsum[wg ^ 1][2][r];
      // Cluster split: the final state merges this CTA's (a_self) and the peer's (a_peer).
      float m_fin = m_all, l_fin = l_all, lx_fin = lx_all, mu_fin = mu_all;
      float a_self = 1.0f, a_peer = 0.0f;
      const uint32_t recv = smem_u32(smem + L::OFF_KDK + kPairRecvOffset);
      const uint32_t recv_row = recv + kPairRecvStats + wg * kPairRecvBlock + r * kPairRecvRowBytes;
      if constexpr (kPair) {
        if (split == 1) {
          // This CTA's state is staged in its own rings (same layout as the
          // peer's receive area) and sent as one bulk copy below.
          if (wg == 0 && JVP_CHECK(kPairRecvOffset + r * 16 + 16 <= L::OFF_CTRL - L::OFF_KDK,
                                   p.status, kChkSmem))
            st_shared_v4(recv + r * 16, __float_as_uint(m_all), __float_as_uint(l_all),
                                    __float_as_uint(lx_all), __float_as_uint(mu_all));
        } else {
          ok = warp_wait<kHint>(&ctrl->peer_ready, 0, p.status, abort);
          if (ok) {
            float4 st;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(st.x), "=f"(st.y), "=f"(st.z), "=f"(st.w)
                         : "r"(recv + r * 16));
            m_fin = fmaxf(m_all, st.x);
            a_self = (m_all == -INFINITY) ? 0.0f : exp2f(m_all - m_fin);
            a_peer = (st.x == -INFINITY) ? 0.0f : exp2f(st.x - m_fin);
            l_fin = a_self * l_all + a_peer * st.y;
            lx_fin = a_self * lx_all + a_peer * st.z;
            mu_fin = a_self * mu_all + a_peer * st.w;
          }
        }
      }
      const float inv_l = (l_fin > 0.0f) ? 1.0f / l_fin : 0.0f;
      const float mu_row = mu_fin * inv_l;
      if (!kWsSplit && !(kPair && split == 1) && row_ok && wg == 0) {
        const long long ridx = (static_cast<long long>(b) * p.H + h) * p.Nq + i;
        if (JVP_CHECK(ridx < static_cast<long long>(BH) * p.Nq, p.status, kChkGlobalRow)) {
          if (p.lse) p.lse[ridx] = (lx_fin > 0.0f) ? (m_fin + log2f(lx_fin)) * kLn2 : -INFINITY;
          if (TANGENT && p.mu) p.mu[ridx] = mu_row;
        }
      }
      const uint32_t own = lane_base + L::TM_A + wg * L::ACC_STRIDE;
      const uint32_t oth = lane_base + L::TM_A + (wg ^ 1) * L::ACC_STRIDE;
      const long long rows = static_cast<long long>(BH) * p.Nq;
      const long long R = static_cast<long long>(split) * rows +
                          (static_cast<long long>(b) * p.H + h) * p.Nq + (row_ok ? i : 0);
      float* acc = kWsSplit
                       ? p.split_ws + static_cast<long long>(p.splits) * rows * 4 + R * (2 * D)
                       : nullptr;
      if (kWsSplit && row_ok && wg == 0 &&
          JVP_CHECK(R < static_cast<long long>(p.splits) * rows, p.status, kChkGlobalRow))
        reinterpret_cast<float4*>(p.split_ws)[R] = make_float4(m_all, l_all, lx_all, mu_all);
      wait_acc();
      // With whole tiles and only warpgroup 0's first tile (or pair) of keys,
      // warpgroup 1's accumulator was never written (its weight is 0, its
      // contents undefined).
      const bool only_acc0 = kAlt && n_kv <= (kPairOwn ? 2 : 1);
#pragma unroll 1
      for (int col = wg * (D / 2); ok && col < (wg + 1) * (D / 2); col += 16) {
        float fa[16], ft[16];
        if (n_kv > 0) {
          uint32_t a0[16], t0[16], a1[16], t1[16];
          const bool cols_ok = JVP_CHECK(
              L::TM_A + L::ACC_STRIDE + (TANGENT ? D : 0) + col + 16 <= L::TM_COLS, p.status, kChkTmem);
          if (cols_ok && TANGENT) {
            tmem_ld16x4(own + col, own + D + col, oth + col, oth + D + col, a0, t0, a1, t1);
          } else if (cols_ok) {
            tmem_ld16x2(own + col, oth + col, a0, a1);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            fa[e] = only_acc0 ? __uint_as_float(wg == 0 ? a0[e] : a1[e])
                              : a_own * __uint_as_float(a0[e]) + a_oth * __uint_as_float(a1[e]);
            ft[e] = TANGENT ? a_own * __uint_as_float(t0[e]) + a_oth * __uint_as_float(t1[e]) : 0.f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) fa[e] = ft[e] = 0.f;
        }
        if (kPair && split == 1) {
          // this CTA's A and T rows (its warpgroup's columns), staged locally
          const int lc = col - wg * (D / 2);  // column within the warpgroup's block
          const bool in_recv = JVP_CHECK(
              kPairRecvOffset + kPairRecvStats + wg * kPairRecvBlock + (r + 1) * kPairRecvRowBytes <=
                  L::OFF_CTRL - L::OFF_KDK && (D / 2 + lc + 16) * 4 <= kPairRecvRowBytes,
              p.status, kChkSmem);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            if (!in_recv) break;
            st_shared_v4(recv_row + (lc + 4 * v4) * 4, __float_as_uint(fa[4 * v4]),
                         __float_as_uint(fa[4 * v4 + 1]), __float_as_uint(fa[4 * v4 + 2]),
                         __float_as_uint(fa[4 * v4 + 3]));
            st_shared_v4(recv_row + (D / 2 + lc + 4 * v4) * 4, __float_as_uint(ft[4 * v4]),
                         __float_as_uint(ft[4 * v4 + 1]), __float_as_uint(ft[4 * v4 + 2]),
                         __float_as_uint(ft[4 * v4 + 3]));
          }
        } else if (kWsSplit) {
          if (row_ok) {
            float4* ad = reinterpret_cast<float4*>(acc + col);
            float4* td = reinterpret_cast<float4*>(acc + D + col);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              ad[v4] = make_float4(fa[4 * v4], fa[4 * v4 + 1], fa[4 * v4 + 2], fa[4 * v4 + 3]);
              if (TANGENT)
                td[v4] = make_float4(ft[4 * v4], ft[4 * v4 + 1], ft[4 * v4 + 2], ft[4 * v4 + 3]);
            }
          }
        } else {
          if (kPair && ok) {
            // merge the peer's A and T (received into this CTA's rings)
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              float4 pa, pt4;
              const int lc = col - wg * (D / 2);
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(pa.x), "=f"(pa.y), "=f"(pa.z), "=f"(pa.w)
                           : "r"(recv_row + (lc + 4 * v4) * 4));
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(pt4.x), "=f"(pt4.y), "=f"(pt4.z), "=f"(pt4.w)
                           : "r"(recv_row + (D / 2 + lc + 4 * v4) * 4));
              fa[4 * v4] = a_self * fa[4 * v4] + a_peer * pa.x;
              fa[4 * v4 + 1] = a_self * fa[4 * v4 + 1] + a_peer * pa.y;
              fa[4 * v4 + 2] = a_self * fa[4 * v4 + 2] + a_peer * pa.z;
              fa[4 * v4 + 3] = a_self * fa[4 * v4 + 3] + a_peer * pa.w;
              ft[4 * v4] = a_self * ft[4 * v4] + a_peer * pt4.x;
              ft[4 * v4 + 1] = a_self * ft[4 * v4 + 1] + a_peer * pt4.y;
              ft[4 * v4 + 2] = a_self * ft[4 * v4 + 2] + a_peer * pt4.z;
              ft[4 * v4 + 3] = a_self * ft[4 * v4 + 3] + a_peer * pt4.w;
            }
          }
          uint32_t po[8], pt[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float o0 = fa[e] * inv_l, o1 = fa[e + 1] * inv_l;
            po[e >> 1] = ElemTraits<T>::pack(o0, o1);
            if (TANGENT)
              pt[e >> 1] = ElemTraits<T>::pack(ft[e] * inv_l - mu_row * o0,
                                               ft[e + 1] * inv_l - mu_row * o1);
          }
          {
            stage_row<2>(o_tile, r, col, po, L::KCH * L::BM * 128, p.status);
            if (TANGENT) {
              stage_row<2>(t_tile, r, col, pt, L::KCH * L::BM * 128, p.status);
            }
          }
        }
      }
      if constexpr (kPair) {
        if (split == 1) {
          // Each warp sends its staged rows to rank 0 (once rank 0's rings
          // are free) as bulk copies that complete on rank 0's barrier; this
          // CTA's shared memory stays valid until then because rank 0 passes
          // the final cluster barrier only after that completion.
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (mbar_wait_cluster(&ctrl->ring_free, 0, abort)) {
              const uint32_t bar = cluster_map(smem_u32(&ctrl->peer_ready), 0);
              const uint32_t rows = recv + kPairRecvStats + wg * kPairRecvBlock +
                                    sub * 32 * kPairRecvRowBytes;
              bulk_copy_to_cluster(cluster_map(rows, 0), rows, 32 * kPairRecvRowBytes, bar);
              if (wg == 0) {
                const uint32_t stats = recv + sub * 32 * 16;
                bulk_copy_to_cluster(cluster_map(stats, 0), stats, 32 * 16, bar);
              }
            } else {
              record_timeout(p.status, abort);
            }
          }
        }
      }
    } else if (kWsSplit && ok) {
      // Split-KV: store this key range's unnormalised state (m, l, lx, mu~,
      // A, T) for the combine kernel.
      const long long rows = static_cast<long long>(BH) * p.Nq;
      const long long R = static_cast<long long>(split) * rows +
                          (static_cast<long long>(b) * p.H + h) * p.Nq + (row_ok ? i : 0);
      if (row_ok && wg == 0 &&
          JVP_CHECK(R < static_cast<long long>(p.splits) * rows, p.status, kChkGlobalRow)) {
        reinterpret_cast<float4*>(p.split_ws)[R] =
            make_float4(m_run, l_run + ctrl->xsum[1][0][r], lx_run + ctrl->xsum[1][1][r],
                        mu_run + ctrl->xsum[1][2][r]);
      }
      float* acc = p.split_ws + static_cast<long long>(p.splits) * rows * 4 + R * (2 * D);
      wait_acc();
#pragma unroll 1
      for (int col = wg * (D / 2); ok && col < (wg + 1) * (D / 2); col += 32) {
        uint32_t a[32], tt[32];
        if (n_kv > 0) {
          const bool cols_ok =
              JVP_CHECK(L::TM_T + col + 32 <= L::TM_COLS, p.status, kChkTmem);
          if (cols_ok && TANGENT) {
            tmem_ld32x2(lane_base + L::TM_A + col, lane_base + L::TM_T + col, a, tt);
          } else if (cols_ok) {
            tmem_ld32(lane_base + L::TM_A + col, a);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = tt[e] = 0u;
        }
        if (row_ok) {
          uint4* ad = reinterpret_cast<uint4*>(acc + col);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            ad[v4] = make_uint4(a[4 * v4], a[4 * v4 + 1], a[4 * v4 + 2], a[4 * v4 + 3]);
          if (TANGENT) {
            uint4* td = reinterpret_cast<uint4*>(acc + D + col);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              td[v4] = make_uint4(tt[4 * v4], tt[4 * v4 + 1], tt[4 * v4 + 2], tt[4 * v4 + 3]);
          }
        }
      }
    } else if (ok) {
      const float l_all = l_run + ctrl->xsum[wg ^ 1][0][r];
      const float lx_all = lx_run + ctrl->xsum[wg ^ 1][1][r];
      const float mu_all = mu_run + ctrl->xsum[wg ^ 1][2][r];
      const float inv_l = (l_all > 0.0f) ? 1.0f / l_all : 0.0f;
      const float mu_row = mu_all * inv_l;
      if (row_ok && wg == 0) {
        const long long ridx = (static_cast<long long>(b) * p.H + h) * p.Nq + i;
        if (JVP_CHECK(ridx < static_cast<long long>(BH) * p.Nq, p.status, kChkGlobalRow)) {
          if (p.lse)
            p.lse[ridx] = (lx_all > 0.0f) ? (m_run + log2f(lx_all)) * kLn2 : -INFINITY;
          if (TANGENT && p.mu) p.mu[ridx] = mu_row;
        }
      }
      wait_acc();
#pragma unroll 1
      for (int col = wg * (D / 2); ok && col < (wg + 1) * (D / 2); col += 32) {
        uint32_t a[32], tt[32];
        if (n_kv > 0) {
          const bool cols_ok =
              JVP_CHECK(L::TM_T + col + 32 <= L::TM_COLS, p.status, kChkTmem);
          if (cols_ok && TANGENT) {
            tmem_ld32x2(lane_base + L::TM_A + col, lane_base + L::TM_T + col, a, tt);
          } else if (cols_ok) {
            tmem_ld32(lane_base + L::TM_A + col, a);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = tt[e] = 0u;
        }
        uint32_t po[16], pt[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float o0 = __uint_as_float(a[e]) * inv_l, o1 = __uint_as_float(a[e + 1]) * inv_l;
          po[e >> 1] = ElemTraits<T>::pack(o0, o1);
          if (TANGENT) {
            const float t0 = __uint_as_float(tt[e]) * inv_l - mu_row * o0;
            const float t1 = __uint_as_float(tt[e + 1]) * inv_l - mu_row * o1;
            pt[e >> 1] = ElemTraits<T>::pack(t0, t1);
          }
        }
        stage_row<4>(o_tile, r, col, po, L::KCH * L::BM * 128, p.status);
        if (TANGENT) stage_row<4>(t_tile, r, col, pt, L::KCH * L::BM * 128, p.status);
      }
    }
    if (!kWsSplit && !(kPair && split == 1) && ok) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->o_staged);
      if (warp == 2 && lane == 0) {
        if (mbar_wait<kHint>(&ctrl->o_staged, 0, abort)) {
          for (int c = 0; c < L::KCH; ++c) {
            tma_store_4d(&maps.o, smem + L::OFF_KDK + c * L::BM * 128, c * 64, q0, h, b);
            if (TANGENT)
              tma_store_4d(&maps.t_o, smem + L::OFF_KDK + (L::KCH + c) * L::BM * 128, c * 64, q0,
                           h, b);
          }
          tma_store_commit();
          tma_store_wait_read();  // the CTA's shared memory stays valid until then
        } else {
          record_timeout(p.status, abort);
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  }
  // Cluster split: neither CTA exits while the other may still reach its
  // shared memory.
  if constexpr (kPair) {
    if (warp != 2) cluster_wait();
    cluster_sync();
  }
}

template <typename T, int D, int MASK, bool TANGENT, int SPLIT>
cudaError_t launch_tc_variant(const TcMaps& maps, const FwdParams& p, cudaStream_t stream) {
  using L = TcLayout<D, TANGENT, tc_mask_tile<D, MASK, TANGENT>()>;
  auto kern = fwd_dual_tc_kernel<T, D, MASK, TANGENT, SPLIT>;
  // The attribute is per device; setting it is idempotent, the mask (shared
  // by host threads) only saves calls.
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_done.load(std::memory_order_relaxed) & (1ull << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done.fetch_or(1ull << dev, std::memory_order_relaxed);
  }
  const long long grid = static_cast<long long>(p.num_q_tiles) * p.B * p.H * (SPLIT ? p.splits : 1);
  if constexpr (SPLIT == kSplitCluster) {
    // the two CTAs of a query tile (consecutive blocks) form a cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(tc_threads<D, MASK, TANGENT, SPLIT>());
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps, p);
  }
  kern<<<static_cast<unsigned>(grid), tc_threads<D, MASK, TANGENT, SPLIT>(), L::SMEM_BYTES,
         stream>>>(maps, p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_tc_dispatch(int mask_kind, bool tangent, const TcMaps& maps,
                               const FwdParams& p, cudaStream_t stream) {
#define JVP_TC_CASE(MK)                                                                  \
  case MK:                                                                               \
    if (!tangent) return launch_tc_variant<T, D, MK, false, 0>(maps, p, stream);         \
    if (p.splits > 1 && p.split_ws)                                                      \
      return launch_tc_variant<T, D, MK, true, kSplitWorkspace>(maps, p, stream);        \
    if (p.splits > 1) {                                                                  \
      if constexpr (D == 64) return launch_tc_variant<T, D, MK, true, kSplitCluster>(maps, p, stream); \
      return cudaErrorInvalidValue;                                                      \
    }                                                                                    \
    return launch_tc_variant<T, D, MK, true, 0>(maps, p, stream);
  switch (mask_kind) {
    JVP_TC_CASE(kMaskNone)
    JVP_TC_CASE(kMaskBool)
    JVP_TC_CASE(kMaskAdditive)
    JVP_TC_CASE(kMaskCausal)
    default:
      return cudaErrorInvalidValue;
  }
#undef JVP_TC_CASE
}

}  // namespace jvp

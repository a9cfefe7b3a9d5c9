// jvp_internal.h -- launch descriptions shared by the host entry points and
// the kernel translation units (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace jvp {

enum DType { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum MaskKind { kMaskNone = 0, kMaskBool = 1, kMaskAdditive = 2, kMaskCausal = 3 };

struct Strides {
  long long b, h, n;  // element strides; d stride is 1
};

// Everything a forward kernel needs besides the tensor maps.
struct FwdParams {
  int B, H, Nq, Nk, D;
  int num_q_tiles;
  int group_heads;   // tensor-core kernel: (batch, head) pairs per scheduling group
  float scale;       // logit scale s
  float scale_log2;  // s * log2(e)
  // Tensor-core kernel with s < 0: the score products are formed negated (the
  // MMA's negate-A bit) and scale, scale_log2 hold |s|, so every later step
  // sees the same scaled logits and tangents as for a positive scale.
  int neg_scores;
  const void* mask;  // uint8 (bool) or float (additive); nullptr otherwise
  long long msb, msh, msq, msk;  // mask element strides
  int mask_vec;      // 1: rows are 16-byte aligned and stride_k == 1 (vector loads)
  int mask_tma;      // 1: TcMaps::msk describes the additive mask (tensor-core kernel, D = 128)
  int causal;        // 1: a bool / additive mask also keeps only keys j <= i
  int kv_group;      // query heads per key/value head (grouped-query attention; 1 = none)
  // Split-KV (tensor-core kernel): `splits` CTAs share a query tile, each over
  // a contiguous range of key tiles, and write partial states to `split_ws`
  // (see SplitLayout) for fwd_combine_kernel; splits == 1 and split_ws ==
  // nullptr for the ordinary single-pass kernel.
  int splits;
  float* split_ws;
  // inputs (used by the CUDA-core kernel; the tensor-core kernel reads them by TMA)
  const void *q, *k, *v, *dq, *dk, *dv;
  Strides sq, sk, sv, sdq, sdk, sdv;
  // outputs
  void* o;
  void* t_o;
  Strides so, sto;
  float* lse;
  float* mu;
  unsigned int* status;  // device status word (timeouts)
};

// Workspace of the split-KV forward: for split sp and query row R =
// (b*H + h)*Nq + i, a float4 {m (log2 units), l (rounded p~ sum), lx (fp32 p~
// sum), mu~} at stats[sp*rows + R], then fp32 A[D] and T[D] at
// acc[(sp*rows + R) * 2D].  Every entry is written before it is read.
struct SplitLayout {
  long long rows;  // B * H * Nq
  int D;
  __host__ __device__ size_t stats_floats() const { return static_cast<size_t>(rows) * 4; }
  __host__ __device__ static size_t bytes(long long rows, int D, int splits) {
    return static_cast<size_t>(splits) * static_cast<size_t>(rows) * (4 + 2 * D) * sizeof(float);
  }
};
// Merge of the split-KV partial states into O, tO, lse and mu (any dtype).
cudaError_t launch_fwd_combine(DType dt, bool tangent, const FwdParams& p, cudaStream_t stream);

// Tensor maps of the tensor-core kernel: q, k, v, dq, dk, dv (tangent maps
// are unused by the primal-only variant).
struct TcMaps {
  CUtensorMap q, k, v, dq, dk, dv;
  CUtensorMap o, t_o;  // outputs, 128-row boxes (the epilogue's TMA stores)
  CUtensorMap msk;     // additive mask [B|1, H|1, Nq, Nk] fp32, {32, 128} boxes (if mask_tma)
};

// Tensor-core kernels (fp16/bf16, D in {64, 128}).  Return a cudaError_t.
cudaError_t launch_fwd_tc(DType dt, int D, int mask_kind, bool tangent, const TcMaps& maps,
                          const FwdParams& p, cudaStream_t stream);
constexpr int kTcBlockM = 128;
constexpr int kTcBlockN = 64;

// CUDA-core kernel (any dtype, D <= 128).
cudaError_t launch_fwd_simt(DType dt, int mask_kind, bool tangent, const FwdParams& p,
                            cudaStream_t stream);

// Per-variant entry points of the tensor-core kernel, one translation unit per
// (dtype, D) so that the build compiles them in parallel.
cudaError_t launch_fwd_tc_f16_d64(int mask_kind, bool tangent, const TcMaps& maps,
                                  const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_tc_f16_d128(int mask_kind, bool tangent, const TcMaps& maps,
                                   const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_tc_bf16_d64(int mask_kind, bool tangent, const TcMaps& maps,
                                   const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_tc_bf16_d128(int mask_kind, bool tangent, const TcMaps& maps,
                                    const FwdParams& p, cudaStream_t stream);

// Everything the backward kernels need.  The workspace holds two float32
// arrays [B, H, Nq]: nu = gtO . O and delta = gO . O + gtO . tO - mu * nu.
struct BwdParams {
  int B, H, Nq, Nk, D;
  float scale;
  int mask_kind;
  int causal;    // 1: a bool / additive mask also keeps only keys j <= i
  int kv_group;  // query heads per key/value head (grouped-query attention; 1 = none)
  const void* mask;
  long long msb, msh, msq, msk;
  int mask_vec;  // 1: mask rows are 16-byte aligned and stride_k == 1 (vector loads)
  const void *q, *k, *v, *dq, *dk, *dv, *o, *t_o, *g_o, *g_to;
  Strides sq, sk, sv, sdq, sdk, sdv, so, sto, sgo, sgto;
  const float* lse;
  const float* mu;
  void *g_q, *g_k, *g_v, *g_dq, *g_dk, *g_dv;
  Strides sgq, sgk, sgv, sgdq, sgdk, sgdv;
  float* nu;
  float* delta;
  // 1: the backward of attention without tangents (dq, dk, dv, t_o, g_to, mu
  // are not read and may be NULL; g_dq, g_dk, g_dv are not written; the row
  // pass stores nu = 0 and delta = gO . O)
  int primal;
  // Key-major split (ksplits > 1): each (batch, key/value head, key tile)'s
  // query tiles are shared by ksplits CTAs, which write fp32 partial sums of
  // (g_dV, gV, g_dK, gK) to kws [ksplits][4][B*Hkv][Nk][D]; a combine kernel
  // adds them into the outputs.
  int ksplits;
  float* kws;
  // Query-major split (qsplits > 1): each (batch, head, query tile)'s key
  // tiles are shared by qsplits CTAs, which write fp32 partial sums of
  // (g_dQ, gQ) to qws [qsplits][2][B*H][Nq][D]; a combine kernel adds them.
  int qsplits;
  float* qws;
};

// Key-major splits of the backward for a problem: >1 when its key-major CTAs
// (B * Hkv * ceil(Nk / 128)) fill less than half of the SMs and each walks
// at least 64 query tiles of 64 rows (grouped-query heads, long sequences);
// every split keeps 32 or more.  (Shorter loops do not repay the partial
// sums' extra traffic and the combine kernel: measured slower.)
inline int bwd_key_splits(long long B, long long Hkv, long long Nq, long long Nk, long long group,
                          int num_sms) {
  const long long ctas = B * Hkv * ((Nk + 127) / 128);
  const long long tiles = ((Nq + 63) / 64) * group;  // query tiles of a CTA (64-row tiles)
  if (ctas <= 0 || 2 * ctas > num_sms || tiles < 64) return 1;
  long long s = num_sms / ctas;
  s = s < 16 ? s : 16;
  s = s < tiles / 32 ? s : tiles / 32;
  return s > 1 ? static_cast<int>(s) : 1;
}
// Query-major splits: the same rule for the query-major CTAs (B * H *
// ceil(Nq / 128)) walking 64 or more key tiles of 64 (few queries, many keys).
inline int bwd_query_splits(long long B, long long H, long long Nq, long long Nk, int num_sms) {
  const long long ctas = B * H * ((Nq + 127) / 128);
  const long long tiles = (Nk + 63) / 64;
  if (ctas <= 0 || 2 * ctas > num_sms || tiles < 64) return 1;
  long long s = num_sms / ctas;
  s = s < 16 ? s : 16;
  s = s < tiles / 32 ? s : tiles / 32;
  return s > 1 ? static_cast<int>(s) : 1;
}
// Bytes of the query-major partial sums for `splits` (0 when not split).
inline size_t bwd_query_split_bytes(int splits, long long B, long long H, long long Nq,
                                    long long D) {
  return splits > 1 ? static_cast<size_t>(splits) * 2 * static_cast<size_t>(B * H * Nq * D) *
                          sizeof(float)
                    : 0;
}
// Bytes of the key-major partial sums for `splits` (0 when not split).
inline size_t bwd_key_split_bytes(int splits, long long B, long long Hkv, long long Nk,
                                  long long D) {
  return splits > 1 ? static_cast<size_t>(splits) * 4 * static_cast<size_t>(B * Hkv * Nk * D) *
                          sizeof(float)
                    : 0;
}

// Workspace bytes of the backward for a problem with `rows` = B * H * Nq query rows.
inline size_t bwd_workspace_bytes(long long rows) {
  return static_cast<size_t>(2 * rows) * sizeof(float);
}

// Backward of the dual computation (CUDA-core kernels).  Returns a cudaError_t.
cudaError_t launch_bwd_simt(DType dt, const BwdParams& p, cudaStream_t stream);
// Only the per-row pre-pass (nu and delta into the workspace).
cudaError_t launch_bwd_rows(DType dt, const BwdParams& p, cudaStream_t stream);

// Tensor maps of the tensor-core backward kernels (query-side and key-side
// tensors; each kernel gets its own set, the box heights differ).
struct BwdTcMaps {
  CUtensorMap q, dq, go, gto, k, dk, v, dv;
  // query-side maps with a second box height (key-major kernel: 64 rows for
  // its value part; the maps above have 32)
  CUtensorMap q64, dq64, go64, gto64;
};
// Tensor-core backward (fp16/bf16, D in {64, 128}; primal: the backward of
// attention without tangents); the row pre-pass must have been enqueued before.  qmaps: query-major kernel (query-side boxes of
// 128 rows, key side 64); kmaps: key-major kernel (key side 128, query side 32).
// The query-major kernel goes to `stream`, the key-major kernel(s) to
// `kstream` (the same stream, or a second one the caller has made wait for
// the row pass and joins back).
cudaError_t launch_bwd_tc(DType dt, int D, int mask_kind, bool primal, const BwdTcMaps& qmaps,
                          const BwdTcMaps& kmaps, const BwdParams& p, int num_sms,
                          unsigned int* status, cudaStream_t stream, cudaStream_t kstream);
#define JVP_BWD_TC_DECL(NAME)                                                            \
  cudaError_t NAME(int mask_kind, const BwdTcMaps& qmaps, const BwdTcMaps& kmaps,        \
                   const BwdParams& p, int num_sms, unsigned int* status,               \
                   cudaStream_t stream, cudaStream_t kstream);
JVP_BWD_TC_DECL(launch_bwd_tc_f16_d64)
JVP_BWD_TC_DECL(launch_bwd_tc_f16_d128)
JVP_BWD_TC_DECL(launch_bwd_tc_bf16_d64)
JVP_BWD_TC_DECL(launch_bwd_tc_bf16_d128)
// The same kernels specialised for the primal backward (p.primal = 1).
JVP_BWD_TC_DECL(launch_bwd_primal_tc_f16_d64)
JVP_BWD_TC_DECL(launch_bwd_primal_tc_f16_d128)
JVP_BWD_TC_DECL(launch_bwd_primal_tc_bf16_d64)
JVP_BWD_TC_DECL(launch_bwd_primal_tc_bf16_d128)
#undef JVP_BWD_TC_DECL

// Device status word owned by the library (bit 0: a bounded wait timed out).
unsigned int* device_status_ptr();

}  // namespace jvp

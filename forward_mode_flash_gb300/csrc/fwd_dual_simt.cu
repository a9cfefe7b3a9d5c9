// fwd_dual_simt.cu -- CUDA-core kernel for attention forward + JVP: fp32 FFMA
// arithmetic for every element type and any head dimension up to 128.  It is
// the path for float32 inputs (whose error budget rules out the tf32 tensor
// kind) and for fp16/bf16 shapes the tensor-core kernel does not take.
//
// Same computation as the tensor-core kernel ("JVP Flash Attention" project
// page, Description and Usage sections): one pass over key chunks with an
// online softmax carrying the running maximum m, row sum l, the running sum
// mu~ of p~ * dS, and the accumulators A = sum p~ V, T = sum p~ (dS V + dV).
//
// Decomposition: one warp per query row, eight rows per 256-thread block.
// Per chunk of 32 keys the block stages K, dK, V, dV (as fp32) in shared
// memory; lane j of each warp forms the scores of key j (S, dQ.K, Q.dK), the
// warp reduces the chunk's maximum and sums with shuffles, then every lane
// accumulates its slice of the head dimension (d = lane + 32u).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "jvp_internal.h"

namespace jvp {
namespace {

constexpr int kRows = 8;     // warps (query rows) per block
constexpr int kChunk = 32;   // keys per staged chunk
constexpr int kMaxU = 4;     // head-dimension elements per lane (D <= 128)

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T, int MASK, bool TANGENT>
__global__ void __launch_bounds__(kRows * 32)
    fwd_dual_simt_kernel(const FwdParams p) {
  extern __shared__ float sm[];
  const int D = p.D;
  const int ld = D + 1;  // padded row: lane-strided reads hit distinct banks
  float* sK = sm;
  float* sV = sK + kChunk * ld;
  float* sdK = sV + kChunk * ld;
  float* sdV = sdK + kChunk * ld;
  float* sQ = sdV + kChunk * ld;  // [kRows][D]
  float* sdQ = sQ + kRows * D;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_row_blocks = (p.Nq + kRows - 1) / kRows;
  const int bh = blockIdx.x % (p.B * p.H);
  int rb = blockIdx.x / (p.B * p.H);
  // Causal alone, or on top of a bool / additive mask (runtime flag).
  const bool causal =
      (MASK == kMaskCausal) || ((MASK == kMaskBool || MASK == kMaskAdditive) && p.causal != 0);
  if (causal) rb = n_row_blocks - 1 - rb;
  const int b = bh / p.H, h = bh % p.H;
  const int hk = h / p.kv_group;  // key/value head (grouped-query attention)
  const int i = rb * kRows + warp;
  const bool row_ok = i < p.Nq;

  const T* q = static_cast<const T*>(p.q) + b * p.sq.b + h * p.sq.h;
  const T* k = static_cast<const T*>(p.k) + b * p.sk.b + hk * p.sk.h;
  const T* v = static_cast<const T*>(p.v) + b * p.sv.b + hk * p.sv.h;
  const T* dq = TANGENT ? static_cast<const T*>(p.dq) + b * p.sdq.b + h * p.sdq.h : nullptr;
  const T* dk = TANGENT ? static_cast<const T*>(p.dk) + b * p.sdk.b + hk * p.sdk.h : nullptr;
  const T* dv = TANGENT ? static_cast<const T*>(p.dv) + b * p.sdv.b + hk * p.sdv.h : nullptr;

  for (int d = lane; d < D; d += 32) {
    sQ[warp * D + d] = row_ok ? to_f32(q[static_cast<long long>(i) * p.sq.n + d]) : 0.f;
    if (TANGENT)
      sdQ[warp * D + d] = row_ok ? to_f32(dq[static_cast<long long>(i) * p.sdq.n + d]) : 0.f;
  }

  int n_keys = p.Nk;
  if (causal) n_keys = min(n_keys, min(rb * kRows + kRows, p.Nq));
  const float* mrow_f = nullptr;
  const uint8_t* mrow_b = nullptr;
  if (row_ok) {
    const long long off = b * p.msb + h * p.msh + static_cast<long long>(i) * p.msq;
    if (MASK == kMaskBool) mrow_b = static_cast<const uint8_t*>(p.mask) + off;
    if (MASK == kMaskAdditive) mrow_f = static_cast<const float*>(p.mask) + off;
  }

  float m_run = -INFINITY, l_run = 0.f, mu_run = 0.f;
  float A[kMaxU], Tacc[kMaxU];
#pragma unroll
  for (int u = 0; u < kMaxU; ++u) A[u] = Tacc[u] = 0.f;

  for (int j0 = 0; j0 < n_keys; j0 += kChunk) {
    __syncthreads();
    const int nj = min(kChunk, n_keys - j0);
    for (int e = threadIdx.x; e < nj * D; e += blockDim.x) {
      const int jj = e / D, d = e % D;
      const long long j = j0 + jj;
      sK[jj * ld + d] = to_f32(k[j * p.sk.n + d]);
      sV[jj * ld + d] = to_f32(v[j * p.sv.n + d]);
      if (TANGENT) {
        sdK[jj * ld + d] = to_f32(dk[j * p.sdk.n + d]);
        sdV[jj * ld + d] = to_f32(dv[j * p.sdv.n + d]);
      }
    }
    __syncthreads();
    if (!row_ok) continue;

    // Scores of key j0 + lane.
    const int j = j0 + lane;
    bool keep = lane < nj;
    float bias = 0.f;
    if (keep) {
      if (MASK == kMaskCausal) keep = j <= i;
      if (MASK == kMaskBool) keep = mrow_b[static_cast<long long>(j) * p.msk] != 0;
      if (MASK == kMaskAdditive) {
        bias = mrow_f[static_cast<long long>(j) * p.msk];
        keep = !(isinf(bias) && bias < 0.f);
      }
      if (MASK != kMaskCausal && causal) keep = keep && j <= i;
    }
    float s_qk = 0.f, s_t = 0.f;
    if (keep) {
      const float* kr = sK + lane * ld;
      const float* dkr = sdK + lane * ld;
      const float* qr = sQ + warp * D;
      const float* dqr = sdQ + warp * D;
      for (int d = 0; d < D; ++d) {
        s_qk = fmaf(qr[d], kr[d], s_qk);
        if (TANGENT) s_t = fmaf(dqr[d], kr[d], fmaf(qr[d], dkr[d], s_t));
      }
    }
    const float x = keep ? fmaf(p.scale, s_qk, bias) : -INFINITY;
    const float m_new = fmaxf(m_run, warp_max(x));
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = (m_run == -INFINITY) ? 0.f : expf(m_run - m_use);
    const float pj = keep ? expf(x - m_use) : 0.f;
    const float pdj = TANGENT ? pj * (p.scale * s_t) : 0.f;
    l_run = l_run * alpha + warp_sum(pj);
    if (TANGENT) mu_run = mu_run * alpha + warp_sum(pdj);
    m_run = m_new;
#pragma unroll
    for (int u = 0; u < kMaxU; ++u) {
      A[u] *= alpha;
      if (TANGENT) Tacc[u] *= alpha;
    }
    for (int jj = 0; jj < nj; ++jj) {
      const float pb = __shfl_sync(0xffffffffu, pj, jj);
      const float pdb = TANGENT ? __shfl_sync(0xffffffffu, pdj, jj) : 0.f;
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) {
        const int d = lane + 32 * u;
        if (d < D) {
          const float vv = sV[jj * ld + d];
          A[u] = fmaf(pb, vv, A[u]);
          if (TANGENT) Tacc[u] = fmaf(pdb, vv, fmaf(pb, sdV[jj * ld + d], Tacc[u]));
        }
      }
    }
  }

  if (!row_ok) return;
  const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
  const float mu_row = mu_run * inv_l;
  T* orow = static_cast<T*>(p.o) + b * p.so.b + h * p.so.h + static_cast<long long>(i) * p.so.n;
  T* trow = TANGENT ? static_cast<T*>(p.t_o) + b * p.sto.b + h * p.sto.h +
                          static_cast<long long>(i) * p.sto.n
                    : nullptr;
#pragma unroll
  for (int u = 0; u < kMaxU; ++u) {
    const int d = lane + 32 * u;
    if (d < D) {
      const float o = A[u] * inv_l;
      orow[d] = from_f32<T>(o);
      if (TANGENT) trow[d] = from_f32<T>(Tacc[u] * inv_l - mu_row * o);
    }
  }
  if (lane == 0) {
    const long long ridx = (static_cast<long long>(b) * p.H + h) * p.Nq + i;
    if (p.lse) p.lse[ridx] = (l_run > 0.f) ? m_run + logf(l_run) : -INFINITY;
    if (TANGENT && p.mu) p.mu[ridx] = mu_row;
  }
}

template <typename T, int MASK, bool TANGENT>
cudaError_t launch_variant(const FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_dual_simt_kernel<T, MASK, TANGENT>;
  const size_t smem = (4 * kChunk * (p.D + 1) + 2 * kRows * p.D) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>((p.Nq + kRows - 1) / kRows) * p.B * p.H;
  kern<<<static_cast<unsigned>(blocks), kRows * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_mask(int mask_kind, bool tangent, const FwdParams& p, cudaStream_t stream) {
#define JVP_SIMT_CASE(MK)                                          \
  case MK:                                                         \
    return tangent ? launch_variant<T, MK, true>(p, stream)        \
                   : launch_variant<T, MK, false>(p, stream);
  switch (mask_kind) {
    JVP_SIMT_CASE(kMaskNone)
    JVP_SIMT_CASE(kMaskBool)
    JVP_SIMT_CASE(kMaskAdditive)
    JVP_SIMT_CASE(kMaskCausal)
    default:
      return cudaErrorInvalidValue;
  }
#undef JVP_SIMT_CASE
}

}  // namespace

cudaError_t launch_fwd_simt(DType dt, int mask_kind, bool tangent, const FwdParams& p,
                            cudaStream_t stream) {
  switch (dt) {
    case kF32:
      return dispatch_mask<float>(mask_kind, tangent, p, stream);
    case kF16:
      return dispatch_mask<__half>(mask_kind, tangent, p, stream);
    case kBF16:
      return dispatch_mask<__nv_bfloat16>(mask_kind, tangent, p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace jvp

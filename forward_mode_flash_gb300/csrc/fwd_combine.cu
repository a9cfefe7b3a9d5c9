// fwd_combine.cu -- merge of split-KV partial states (the associative merge of
// online-softmax states: each key range contributes (m, l, lx, mu~, A, T)
// relative to its own running max m; with M = max m_s and a_s = 2^(m_s - M),
// l = sum a_s l_s, mu~ = sum a_s mu~_s, A = sum a_s A_s, T = sum a_s T_s), then
// the same normalisation as the single-pass epilogue:
//   O = A / l,  mu = mu~ / l,  tO = T / l - mu O,  lse = (M + log2 lx) ln 2.
// One warp per query row; lane L owns D/32 consecutive columns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "jvp_internal.h"

namespace jvp {
namespace {

constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ void store(__half* p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void store(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store(float* p, float x) { *p = x; }

template <typename T, bool TANGENT, int PER>
__global__ void __launch_bounds__(kRowsPerBlock * 32) fwd_combine_kernel(const FwdParams p) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  const long long R = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (R >= rows) return;
  const int D = p.D;
  const float4* stats = reinterpret_cast<const float4*>(p.split_ws);
  const float* accb = p.split_ws + static_cast<long long>(p.splits) * rows * 4;

  float M = -INFINITY;
  for (int sp = 0; sp < p.splits; ++sp) M = fmaxf(M, stats[sp * rows + R].x);
  float l = 0.f, lx = 0.f, mu = 0.f;
  float a[PER], t[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) a[e] = t[e] = 0.f;
  if (M != -INFINITY) {
    for (int sp = 0; sp < p.splits; ++sp) {
      const float4 st = stats[sp * rows + R];
      if (st.x == -INFINITY) continue;  // empty or fully excluded key range (warp-uniform)
      const float w = exp2f(st.x - M);
      l = fmaf(w, st.y, l);
      lx = fmaf(w, st.z, lx);
      mu = fmaf(w, st.w, mu);
      const float* acc = accb + (sp * rows + R) * (2 * D) + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        a[e] = fmaf(w, acc[e], a[e]);
        if (TANGENT) t[e] = fmaf(w, acc[D + e], t[e]);
      }
    }
  }
  const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
  const float mu_row = mu * inv_l;
  const int b = static_cast<int>(R / (static_cast<long long>(p.H) * p.Nq));
  const int h = static_cast<int>((R / p.Nq) % p.H);
  const int i = static_cast<int>(R % p.Nq);
  T* orow = static_cast<T*>(p.o) + static_cast<long long>(b) * p.so.b +
            static_cast<long long>(h) * p.so.h + static_cast<long long>(i) * p.so.n + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const float o = a[e] * inv_l;
    store(orow + e, o);
    if (TANGENT) {
      T* trow = static_cast<T*>(p.t_o) + static_cast<long long>(b) * p.sto.b +
                static_cast<long long>(h) * p.sto.h + static_cast<long long>(i) * p.sto.n +
                lane * PER;
      store(trow + e, t[e] * inv_l - mu_row * o);
    }
  }
  if (lane == 0) {
    if (p.lse) p.lse[R] = (lx > 0.0f) ? (M + log2f(lx)) * 0.6931471805599453f : -INFINITY;
    if (TANGENT && p.mu) p.mu[R] = mu_row;
  }
}

template <typename T, bool TANGENT>
cudaError_t launch_t(const FwdParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks == 0) return cudaSuccess;
  if (p.D == 64) {
    fwd_combine_kernel<T, TANGENT, 2>
        <<<static_cast<unsigned>(blocks), kRowsPerBlock * 32, 0, stream>>>(p);
  } else if (p.D == 128) {
    fwd_combine_kernel<T, TANGENT, 4>
        <<<static_cast<unsigned>(blocks), kRowsPerBlock * 32, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_combine(DType dt, bool tangent, const FwdParams& p, cudaStream_t stream) {
  if (dt == kF16) return tangent ? launch_t<__half, true>(p, stream) : launch_t<__half, false>(p, stream);
  if (dt == kBF16)
    return tangent ? launch_t<__nv_bfloat16, true>(p, stream)
                   : launch_t<__nv_bfloat16, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace jvp

// bwd_dual_simt.cu -- reverse mode of the dual computation (the backward that
// training through fwd_dual and Hessian-vector products need: the "JVP Flash
// Attention" project page, Description (JVPs and HVPs) and Results (training
// with fwd_dual matches SDPA's loss)).  CUDA-core kernels, fp32 arithmetic.
//
// Given the cotangents gO, gtO of Loss = <gO, O> + <gtO, tO>, per (b, h):
//   P   = exp(S - lse)           S  = s Q K^T + M        dS = s (dQ K^T + Q dK^T)
//   dP  = P * (dS - mu)          (the tangent of P; mu = rowsum(P * dS))
//   G   = gtO V^T                nu = rowsum(gtO * O)
//   gP  = gO V^T + gtO dV^T + G * (dS - mu) - nu * dS
//   delta = rowsum(P * gP) = gO . O + gtO . tO - mu * nu
//   gS  = P * (gP - delta)       g_dS = P * (G - nu)
//   gQ  = s (gS K + g_dS dK)     g_dQ = s g_dS K
//   gK  = s (gS^T Q + g_dS^T dQ) g_dK = s g_dS^T Q
//   gV  = P^T gO + dP^T gtO      g_dV = P^T gtO
// (no gradient reaches the mask).  Each (i, j) term is recomputed from the
// saved lse and mu, so nothing of size N x N is stored.
//
// The same kernels serve the backward of attention without tangents
// (p.primal: dQ = dK = dV = gtO = 0, so nu = 0, delta = gO . O and only gQ,
// gK, gV are written).
//
// Three kernels on the caller's stream:
//   1. rows:   nu and delta per query row, into the workspace;
//   2. keys:   one thread group per key (16 head-dim elements per thread),
//              streaming query rows through shared memory; accumulates gK,
//              g_dK, gV, g_dV in registers and writes them once;
//   3. queries: the mirror image for gQ and g_dQ, streaming key rows.
// No atomics; kernels 2 and 3 both recompute the six score products.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "jvp_internal.h"

namespace jvp {
namespace {

constexpr int kThreads = 256;
constexpr int kPart = 16;    // head-dimension elements per thread
constexpr int kChunk = 32;   // rows staged in shared memory per step

template <typename T>
__device__ __forceinline__ float ld(const T* p);
template <>
__device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld<__half>(const __half* p) { return __half2float(*p); }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st(T* p, float x);
template <>
__device__ __forceinline__ void st<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st<__half>(__half* p, float x) { *p = __float2half_rn(x); }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

template <typename T>
__device__ __forceinline__ const T* row_ptr(const void* base, const Strides& s, int b, int h,
                                            int n) {
  return static_cast<const T*>(base) + b * s.b + h * s.h + static_cast<long long>(n) * s.n;
}

// Sum over the `width` consecutive lanes that share one key (or row).
__device__ __forceinline__ float group_sum(float x, int width) {
  for (int o = 1; o < width; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Causal alone, or on top of a bool / additive mask.
__device__ __forceinline__ bool is_causal(const BwdParams& p) {
  return p.mask_kind == kMaskCausal || p.causal != 0;
}

// Whether key j takes part in row i, and the additive bias.
__device__ __forceinline__ bool keep_ij(const BwdParams& p, int b, int h, int i, int j,
                                        float* bias) {
  *bias = 0.f;
  if (p.causal && j > i) return false;
  switch (p.mask_kind) {
    case kMaskCausal:
      return j <= i;
    case kMaskBool:
      return static_cast<const uint8_t*>(p.mask)[b * p.msb + h * p.msh +
                                                 static_cast<long long>(i) * p.msq +
                                                 static_cast<long long>(j) * p.msk] != 0;
    case kMaskAdditive: {
      const float x = static_cast<const float*>(p.mask)[b * p.msb + h * p.msh +
                                                        static_cast<long long>(i) * p.msq +
                                                        static_cast<long long>(j) * p.msk];
      *bias = x;
      return !(isinf(x) && x < 0.f);
    }
    default:
      return true;
  }
}

// Shared-memory position of head-dim element d of a staged row: the 16
// elements of thread part pp are spread as four float4 groups interleaved
// across parts, so a warp's float4 reads of one row hit distinct banks.
__device__ __forceinline__ int sm_pos(int d, int parts) {
  const int pp = d / kPart, e = d % kPart;
  return ((e >> 2) * parts + pp) * 4 + (e & 3);
}

// ------------------------------------------------------------------ kernel 1
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_rows_kernel(BwdParams p) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  if (warp >= rows) return;
  const int i = warp % p.Nq, bh = warp / p.Nq, b = bh / p.H, h = bh % p.H;
  const T* o = row_ptr<T>(p.o, p.so, b, h, i);
  const T* go = row_ptr<T>(p.g_o, p.sgo, b, h, i);
  float nu = 0.f, a = 0.f;
  if (p.primal) {  // no tangents: nu = 0, delta = gO . O
    for (int d = lane; d < p.D; d += 32) a = fmaf(ld(go + d), ld(o + d), a);
  } else {
    const T* to = row_ptr<T>(p.t_o, p.sto, b, h, i);
    const T* gto = row_ptr<T>(p.g_to, p.sgto, b, h, i);
    for (int d = lane; d < p.D; d += 32) {
      const float od = ld(o + d), gtod = ld(gto + d);
      nu = fmaf(gtod, od, nu);
      a = fmaf(ld(go + d), od, fmaf(gtod, ld(to + d), a));
    }
  }
  for (int off = 16; off > 0; off >>= 1) {
    nu += __shfl_xor_sync(0xffffffffu, nu, off);
    a += __shfl_xor_sync(0xffffffffu, a, off);
  }
  if (lane == 0) {
    p.nu[warp] = nu;
    p.delta[warp] = p.primal ? a : a - p.mu[warp] * nu;
  }
}

// Kernel 1 with 16-byte loads: LPR lanes per row, each reading 16 bytes of
// O, gO (and tO, gtO) — for 16-byte aligned rows whose head dimension is
// LPR * 16 bytes (the tensor-core shapes and fp32 at D = 16..128).
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float (&f)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<__half>(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
    f[2 * k] = t.x; f[2 * k + 1] = t.y;
  }
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

template <typename T, int LPR>
__global__ void __launch_bounds__(kThreads) bwd_rows_vec_kernel(BwdParams p) {
  constexpr int VEC = 16 / sizeof(T);
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gt / LPR;
  const int part = static_cast<int>(gt % LPR);
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  const bool ok = row < rows;  // every lane takes part in the shuffles below
  float nu = 0.f, a = 0.f;
  if (ok) {
    const int i = static_cast<int>(row % p.Nq);
    const long long bh = row / p.Nq;
    const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
    auto ld16 = [&](const void* base, const Strides& st) {
      return *reinterpret_cast<const uint4*>(row_ptr<T>(base, st, b, h, i) + part * VEC);
    };
    float o[VEC], go[VEC];
    unpack16<T>(ld16(p.o, p.so), o);
    unpack16<T>(ld16(p.g_o, p.sgo), go);
#pragma unroll
    for (int e = 0; e < VEC; ++e) a = fmaf(go[e], o[e], a);
    if (!p.primal) {
      float to[VEC], gto[VEC];
      unpack16<T>(ld16(p.t_o, p.sto), to);
      unpack16<T>(ld16(p.g_to, p.sgto), gto);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        nu = fmaf(gto[e], o[e], nu);
        a = fmaf(gto[e], to[e], a);
      }
    }
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) {
    nu += __shfl_xor_sync(0xffffffffu, nu, off);
    a += __shfl_xor_sync(0xffffffffu, a, off);
  }
  if (ok && part == 0) {
    p.nu[row] = nu;
    p.delta[row] = p.primal ? a : a - p.mu[row] * nu;
  }
}

// Per (row i, key j) scalars shared by kernels 2 and 3.
struct PairTerms {
  float P, dP, gS, gdS;
};

__device__ __forceinline__ PairTerms pair_terms(const BwdParams& p, float s_qk, float s_t,
                                                float g, float gp1, float bias, float lse,
                                                float mu, float nu, float delta) {
  PairTerms r;
  const float S = fmaf(p.scale, s_qk, bias);
  r.P = expf(S - lse);
  const float dS = p.scale * s_t;
  r.dP = r.P * (dS - mu);
  const float gP = gp1 + g * (dS - mu) - nu * dS;
  r.gS = r.P * (gP - delta);
  r.gdS = r.P * (g - nu);
  return r;
}

// ------------------------------------------------------------------ kernel 2
// Thread group of `parts` lanes per key; each lane holds 16 head-dim elements.
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_keys_kernel(BwdParams p, int parts) {
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const int stride = parts * kPart;  // floats per staged row
  float* sQ = sm;
  float* sdQ = sQ + kChunk * stride;
  float* sgO = sdQ + kChunk * stride;
  float* sgtO = sgO + kChunk * stride;
  float* sRow = sgtO + kChunk * stride;  // [4][kChunk]: lse, mu, nu, delta

  const int keys_per_block = kThreads / parts;
  const int n_blocks = (p.Nk + keys_per_block - 1) / keys_per_block;
  const int Hkv = p.H / p.kv_group;
  const int bhk = blockIdx.x / n_blocks;  // (batch, key/value head)
  const int kb = blockIdx.x % n_blocks;
  const int b = bhk / Hkv, hk = bhk % Hkv;
  const int part = threadIdx.x % parts;
  const int j = kb * keys_per_block + threadIdx.x / parts;
  const bool key_ok = j < p.Nk;
  const int D = p.D;

  float k_[kPart], dk_[kPart], v_[kPart], dv_[kPart];
  float gk[kPart], gdk[kPart], gv[kPart], gdv[kPart];
#pragma unroll
  for (int e = 0; e < kPart; ++e) {
    const int d = part * kPart + e;
    const bool in = key_ok && d < D;
    const bool tin = in && !p.primal;  // tangent inputs (absent in the primal)
    k_[e] = in ? ld(row_ptr<T>(p.k, p.sk, b, hk, j) + d) : 0.f;
    dk_[e] = tin ? ld(row_ptr<T>(p.dk, p.sdk, b, hk, j) + d) : 0.f;
    v_[e] = in ? ld(row_ptr<T>(p.v, p.sv, b, hk, j) + d) : 0.f;
    dv_[e] = tin ? ld(row_ptr<T>(p.dv, p.sdv, b, hk, j) + d) : 0.f;
    gk[e] = gdk[e] = gv[e] = gdv[e] = 0.f;
  }

  // Causal: rows before the block's first key keep none of its keys.
  const int i_begin = is_causal(p) ? kb * keys_per_block : 0;
  // Grouped-query attention: the key/value head serves kv_group query heads,
  // whose contributions all add into its gradients.
  for (int h = hk * p.kv_group; h < (hk + 1) * p.kv_group; ++h) {
  const long long rbase = (static_cast<long long>(b) * p.H + h) * p.Nq;
  for (int i0 = i_begin; i0 < p.Nq; i0 += kChunk) {
    const int ni = min(kChunk, p.Nq - i0);
    __syncthreads();
    for (int x = threadIdx.x; x < ni * D; x += blockDim.x) {
      const int r = x / D, d = x % D, at = r * stride + sm_pos(d, parts);
      sQ[at] = ld(row_ptr<T>(p.q, p.sq, b, h, i0 + r) + d);
      sdQ[at] = p.primal ? 0.f : ld(row_ptr<T>(p.dq, p.sdq, b, h, i0 + r) + d);
      sgO[at] = ld(row_ptr<T>(p.g_o, p.sgo, b, h, i0 + r) + d);
      sgtO[at] = p.primal ? 0.f : ld(row_ptr<T>(p.g_to, p.sgto, b, h, i0 + r) + d);
    }
    for (int x = threadIdx.x; x < stride * kChunk; x += blockDim.x) {
      // zero the padding of head dims beyond D so partial dots ignore it
      const int r = x / stride, q = x % stride;
      const int pp = (q / 4) % parts, e = ((q / 4) / parts) * 4 + (q & 3);
      if (pp * kPart + e >= D) sQ[x] = sdQ[x] = sgO[x] = sgtO[x] = 0.f;
      (void)r;
    }
    for (int r = threadIdx.x; r < ni; r += blockDim.x) {
      sRow[r] = p.lse[rbase + i0 + r];
      sRow[kChunk + r] = p.primal ? 0.f : p.mu[rbase + i0 + r];
      sRow[2 * kChunk + r] = p.nu[rbase + i0 + r];
      sRow[3 * kChunk + r] = p.delta[rbase + i0 + r];
    }
    __syncthreads();
    for (int r = 0; r < ni; ++r) {
      const int i = i0 + r;
      float q_[kPart], dq_[kPart], go_[kPart], gto_[kPart];
      const float4* q4 = reinterpret_cast<const float4*>(sQ + r * stride);
      const float4* dq4 = reinterpret_cast<const float4*>(sdQ + r * stride);
      const float4* go4 = reinterpret_cast<const float4*>(sgO + r * stride);
      const float4* gto4 = reinterpret_cast<const float4*>(sgtO + r * stride);
#pragma unroll
      for (int g = 0; g < kPart / 4; ++g) {
        const float4 a = q4[g * parts + part], bq = dq4[g * parts + part];
        const float4 c = go4[g * parts + part], dd = gto4[g * parts + part];
        q_[4 * g] = a.x; q_[4 * g + 1] = a.y; q_[4 * g + 2] = a.z; q_[4 * g + 3] = a.w;
        dq_[4 * g] = bq.x; dq_[4 * g + 1] = bq.y; dq_[4 * g + 2] = bq.z; dq_[4 * g + 3] = bq.w;
        go_[4 * g] = c.x; go_[4 * g + 1] = c.y; go_[4 * g + 2] = c.z; go_[4 * g + 3] = c.w;
        gto_[4 * g] = dd.x; gto_[4 * g + 1] = dd.y; gto_[4 * g + 2] = dd.z; gto_[4 * g + 3] = dd.w;
      }
      float s_qk = 0.f, s_t = 0.f, g = 0.f, gp1 = 0.f;
#pragma unroll
      for (int e = 0; e < kPart; ++e) {
        s_qk = fmaf(q_[e], k_[e], s_qk);
        s_t = fmaf(dq_[e], k_[e], fmaf(q_[e], dk_[e], s_t));
        g = fmaf(gto_[e], v_[e], g);
        gp1 = fmaf(go_[e], v_[e], fmaf(gto_[e], dv_[e], gp1));
      }
      s_qk = group_sum(s_qk, parts);
      s_t = group_sum(s_t, parts);
      g = group_sum(g, parts);
      gp1 = group_sum(gp1, parts);
      const float lse = sRow[r];
      float bias;
      if (!key_ok || lse == -INFINITY || !keep_ij(p, b, h, i, j, &bias)) continue;
      const PairTerms t = pair_terms(p, s_qk, s_t, g, gp1, bias, lse, sRow[kChunk + r],
                                     sRow[2 * kChunk + r], sRow[3 * kChunk + r]);
      const float sgS = p.scale * t.gS, sgdS = p.scale * t.gdS;
#pragma unroll
      for (int e = 0; e < kPart; ++e) {
        gv[e] = fmaf(t.P, go_[e], fmaf(t.dP, gto_[e], gv[e]));
        gdv[e] = fmaf(t.P, gto_[e], gdv[e]);
        gk[e] = fmaf(sgS, q_[e], fmaf(sgdS, dq_[e], gk[e]));
        gdk[e] = fmaf(sgdS, q_[e], gdk[e]);
      }
    }
  }
  }  // query heads of the group
  if (!key_ok) return;
#pragma unroll
  for (int e = 0; e < kPart; ++e) {
    const int d = part * kPart + e;
    if (d < D) {
      st(static_cast<T*>(p.g_k) + b * p.sgk.b + hk * p.sgk.h + static_cast<long long>(j) * p.sgk.n + d, gk[e]);
      st(static_cast<T*>(p.g_v) + b * p.sgv.b + hk * p.sgv.h + static_cast<long long>(j) * p.sgv.n + d, gv[e]);
      if (!p.primal) {
        st(static_cast<T*>(p.g_dk) + b * p.sgdk.b + hk * p.sgdk.h + static_cast<long long>(j) * p.sgdk.n + d, gdk[e]);
        st(static_cast<T*>(p.g_dv) + b * p.sgdv.b + hk * p.sgdv.h + static_cast<long long>(j) * p.sgdv.n + d, gdv[e]);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel 3
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_queries_kernel(BwdParams p, int parts) {
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const int stride = parts * kPart;
  float* sK = sm;
  float* sdK = sK + kChunk * stride;
  float* sV = sdK + kChunk * stride;
  float* sdV = sV + kChunk * stride;

  const int rows_per_block = kThreads / parts;
  const int n_blocks = (p.Nq + rows_per_block - 1) / rows_per_block;
  const int bh = blockIdx.x / n_blocks;
  const int qb = blockIdx.x % n_blocks;
  const int b = bh / p.H, h = bh % p.H;
  const int hk = h / p.kv_group;  // key/value head (grouped-query attention)
  const int part = threadIdx.x % parts;
  const int i = qb * rows_per_block + threadIdx.x / parts;
  const bool row_ok = i < p.Nq;
  const int D = p.D;
  const long long ridx = static_cast<long long>(bh) * p.Nq + (row_ok ? i : 0);
  const float lse = row_ok ? p.lse[ridx] : -INFINITY;
  const float mu = (row_ok && !p.primal) ? p.mu[ridx] : 0.f;
  const float nu = row_ok ? p.nu[ridx] : 0.f;
  const float delta = row_ok ? p.delta[ridx] : 0.f;

  float q_[kPart], dq_[kPart], go_[kPart], gto_[kPart], gq[kPart], gdq[kPart];
#pragma unroll
  for (int e = 0; e < kPart; ++e) {
    const int d = part * kPart + e;
    const bool in = row_ok && d < D;
    const bool tin = in && !p.primal;  // tangent inputs (absent in the primal)
    q_[e] = in ? ld(row_ptr<T>(p.q, p.sq, b, h, i) + d) : 0.f;
    dq_[e] = tin ? ld(row_ptr<T>(p.dq, p.sdq, b, h, i) + d) : 0.f;
    go_[e] = in ? ld(row_ptr<T>(p.g_o, p.sgo, b, h, i) + d) : 0.f;
    gto_[e] = tin ? ld(row_ptr<T>(p.g_to, p.sgto, b, h, i) + d) : 0.f;
    gq[e] = gdq[e] = 0.f;
  }

  int j_end = p.Nk;
  if (is_causal(p)) j_end = min(j_end, min(p.Nq, (qb + 1) * rows_per_block));
  for (int j0 = 0; j0 < j_end; j0 += kChunk) {
    const int nj = min(kChunk, j_end - j0);
    __syncthreads();
    for (int x = threadIdx.x; x < nj * D; x += blockDim.x) {
      const int r = x / D, d = x % D, at = r * stride + sm_pos(d, parts);
      sK[at] = ld(row_ptr<T>(p.k, p.sk, b, hk, j0 + r) + d);
      sdK[at] = p.primal ? 0.f : ld(row_ptr<T>(p.dk, p.sdk, b, hk, j0 + r) + d);
      sV[at] = ld(row_ptr<T>(p.v, p.sv, b, hk, j0 + r) + d);
      sdV[at] = p.primal ? 0.f : ld(row_ptr<T>(p.dv, p.sdv, b, hk, j0 + r) + d);
    }
    for (int x = threadIdx.x; x < stride * kChunk; x += blockDim.x) {
      const int q = x % stride;
      const int pp = (q / 4) % parts, e = ((q / 4) / parts) * 4 + (q & 3);
      if (pp * kPart + e >= D) sK[x] = sdK[x] = sV[x] = sdV[x] = 0.f;
    }
    __syncthreads();
    for (int r = 0; r < nj; ++r) {
      const int j = j0 + r;
      float k_[kPart], dk_[kPart], v_[kPart], dv_[kPart];
      const float4* k4 = reinterpret_cast<const float4*>(sK + r * stride);
      const float4* dk4 = reinterpret_cast<const float4*>(sdK + r * stride);
      const float4* v4 = reinterpret_cast<const float4*>(sV + r * stride);
      const float4* dv4 = reinterpret_cast<const float4*>(sdV + r * stride);
#pragma unroll
      for (int g = 0; g < kPart / 4; ++g) {
        const float4 a = k4[g * parts + part], bk = dk4[g * parts + part];
        const float4 c = v4[g * parts + part], dd = dv4[g * parts + part];
        k_[4 * g] = a.x; k_[4 * g + 1] = a.y; k_[4 * g + 2] = a.z; k_[4 * g + 3] = a.w;
        dk_[4 * g] = bk.x; dk_[4 * g + 1] = bk.y; dk_[4 * g + 2] = bk.z; dk_[4 * g + 3] = bk.w;
        v_[4 * g] = c.x; v_[4 * g + 1] = c.y; v_[4 * g + 2] = c.z; v_[4 * g + 3] = c.w;
        dv_[4 * g] = dd.x; dv_[4 * g + 1] = dd.y; dv_[4 * g + 2] = dd.z; dv_[4 * g + 3] = dd.w;
      }
      float s_qk = 0.f, s_t = 0.f, g = 0.f, gp1 = 0.f;
#pragma unroll
      for (int e = 0; e < kPart; ++e) {
        s_qk = fmaf(q_[e], k_[e], s_qk);
        s_t = fmaf(dq_[e], k_[e], fmaf(q_[e], dk_[e], s_t));
        g = fmaf(gto_[e], v_[e], g);
        gp1 = fmaf(go_[e], v_[e], fmaf(gto_[e], dv_[e], gp1));
      }
      s_qk = group_sum(s_qk, parts);
      s_t = group_sum(s_t, parts);
      g = group_sum(g, parts);
      gp1 = group_sum(gp1, parts);
      float bias;
      if (!row_ok || lse == -INFINITY || !keep_ij(p, b, h, i, j, &bias)) continue;
      const PairTerms t = pair_terms(p, s_qk, s_t, g, gp1, bias, lse, mu, nu, delta);
      const float sgS = p.scale * t.gS, sgdS = p.scale * t.gdS;
#pragma unroll
      for (int e = 0; e < kPart; ++e) {
        gq[e] = fmaf(sgS, k_[e], fmaf(sgdS, dk_[e], gq[e]));
        gdq[e] = fmaf(sgdS, k_[e], gdq[e]);
      }
    }
  }
  if (!row_ok) return;
#pragma unroll
  for (int e = 0; e < kPart; ++e) {
    const int d = part * kPart + e;
    if (d < D) {
      st(static_cast<T*>(p.g_q) + b * p.sgq.b + h * p.sgq.h + static_cast<long long>(i) * p.sgq.n + d, gq[e]);
      if (!p.primal)
        st(static_cast<T*>(p.g_dq) + b * p.sgdq.b + h * p.sgdq.h + static_cast<long long>(i) * p.sgdq.n + d, gdq[e]);
    }
  }
}

// Whether every row that kernel 1 reads starts on a 16-byte boundary.
inline bool rows_aligned16(const void* base, const Strides& s, size_t e) {
  return reinterpret_cast<uintptr_t>(base) % 16 == 0 && (s.b * static_cast<long long>(e)) % 16 == 0 &&
         (s.h * static_cast<long long>(e)) % 16 == 0 && (s.n * static_cast<long long>(e)) % 16 == 0;
}

template <typename T, int LPR>
cudaError_t launch_rows_vec(const BwdParams& p, long long rows, cudaStream_t stream) {
  const long long blocks = (rows * LPR + kThreads - 1) / kThreads;
  bwd_rows_vec_kernel<T, LPR><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rows_only(const BwdParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  const long long row_blocks = (rows * 32 + kThreads - 1) / kThreads;
  if (row_blocks == 0) return cudaSuccess;
  // 16-byte loads when the rows allow them: a row of D elements is D * e / 16
  // lanes (2 to 32, a power of two).
  constexpr size_t e = sizeof(T);
  const int lpr = static_cast<int>(p.D * e / 16);
  bool vec = (p.D * e) % 16 == 0 && lpr >= 2 && lpr <= 32 && (lpr & (lpr - 1)) == 0 &&
             rows_aligned16(p.o, p.so, e) && rows_aligned16(p.g_o, p.sgo, e);
  if (vec && !p.primal)
    vec = rows_aligned16(p.t_o, p.sto, e) && rows_aligned16(p.g_to, p.sgto, e);
  if (vec) {
    switch (lpr) {
      case 2: return launch_rows_vec<T, 2>(p, rows, stream);
      case 4: return launch_rows_vec<T, 4>(p, rows, stream);
      case 8: return launch_rows_vec<T, 8>(p, rows, stream);
      case 16: return launch_rows_vec<T, 16>(p, rows, stream);
      case 32: return launch_rows_vec<T, 32>(p, rows, stream);
    }
  }
  bwd_rows_kernel<T><<<static_cast<unsigned>(row_blocks), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_all(const BwdParams& p, cudaStream_t stream) {
  cudaError_t e = launch_rows_only<T>(p, stream);  // (no launch when there are no rows)
  if (e != cudaSuccess) return e;
  // Lanes per key / row: enough 16-element parts to cover D (a power of two).
  int parts = 1;
  while (parts * kPart < p.D) parts <<= 1;
  const size_t smem_k = (4 * kChunk * parts * kPart + 4 * kChunk) * sizeof(float);
  const size_t smem_q = (4 * kChunk * parts * kPart) * sizeof(float);
  e = cudaFuncSetAttribute(bwd_keys_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_k));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_queries_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_q));
  if (e != cudaSuccess) return e;
  const long long per_block = kThreads / parts;
  const long long kblocks =
      static_cast<long long>(p.B) * (p.H / p.kv_group) * ((p.Nk + per_block - 1) / per_block);
  const long long qblocks = static_cast<long long>(p.B) * p.H * ((p.Nq + per_block - 1) / per_block);
  if (kblocks > 0) {
    bwd_keys_kernel<T><<<static_cast<unsigned>(kblocks), kThreads, smem_k, stream>>>(p, parts);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (qblocks > 0) {
    bwd_queries_kernel<T><<<static_cast<unsigned>(qblocks), kThreads, smem_q, stream>>>(p, parts);
    e = cudaGetLastError();
  }
  return e;
}



}  // namespace

cudaError_t launch_bwd_rows(DType dt, const BwdParams& p, cudaStream_t stream) {
  switch (dt) {
    case kF32:
      return launch_rows_only<float>(p, stream);
    case kF16:
      return launch_rows_only<__half>(p, stream);
    case kBF16:
      return launch_rows_only<__nv_bfloat16>(p, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_simt(DType dt, const BwdParams& p, cudaStream_t stream) {
  switch (dt) {
    case kF32:
      return launch_all<float>(p, stream);
    case kF16:
      return launch_all<__half>(p, stream);
    case kBF16:
      return launch_all<__nv_bfloat16>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace jvp

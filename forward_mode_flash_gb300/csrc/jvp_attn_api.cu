// jvp_attn_api.cu -- the C ABI declared in include/jvp_attn.h: argument
// validation, path selection (tensor-core or CUDA-core kernel), TMA tensor-map
// encoding and the device status word.  All compute runs in the kernels; this
// file only checks, describes and enqueues.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <initializer_list>
#include <mutex>
#include <string>

#include "jvp_attn.h"
#include "jvp_internal.h"
#include "sm103_ptx.cuh"

namespace jvp {

// Bit 0: some bounded device wait ran out.  One word per device (each device
// that loads the library gets its own copy of this variable).
__device__ unsigned int g_device_status = 0;

namespace {

thread_local std::string t_last_error;
// 0 none, 1 tensor-core, 2 CUDA-core, 3 tensor-core split-KV (workspace and
// merge kernel), 4 tensor-core split between the two CTAs of a cluster
thread_local int t_last_path = 0;
std::atomic<int> g_cluster_split{1};  // diagnostic switch: 0 never splits across a cluster

jvp_status_t fail(jvp_status_t s, const std::string& msg) {
  t_last_error = msg;
  return s;
}

jvp_status_t ok() {
  t_last_error.clear();
  return JVP_OK;
}

size_t elem_size(int dt) { return dt == JVP_F32 ? 4 : 2; }

// The kernels index sizes and grid dimensions with 32-bit ints.
constexpr int64_t kMaxDim = (1ll << 31) - 1;

// Product of non-negative sizes into *out; false if it overflows int64.
bool checked_product(std::initializer_list<int64_t> xs, int64_t* out) {
  int64_t p = 1;
  for (int64_t x : xs)
    if (__builtin_mul_overflow(p, x, &p)) return false;
  *out = p;
  return true;
}

// Every size of the shape record is at most kMaxDim (checked before any
// product of them is formed).
bool dims_in_range(const jvp_shape_t* s) {
  return s->B <= kMaxDim && s->H <= kMaxDim && s->Nq <= kMaxDim && s->Nk <= kMaxDim &&
         s->D <= kMaxDim && s->Hkv <= kMaxDim;
}

struct DeviceInfo {
  bool queried = false;
  bool sm103 = false;
  int num_sms = 0;
  unsigned int* status = nullptr;
  cudaStream_t side = nullptr;  // the backward's key-side kernels (created on first use)
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

// Looks up (once per device) whether the current device is an sm_103 part
// and where its status word lives.
jvp_status_t current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(JVP_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(JVP_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.queried) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess)
      return fail(JVP_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    d.sm103 = (major == 10 && minor == 3);
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
      return fail(JVP_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_device_status);
    if (e != cudaSuccess)
      return fail(JVP_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    d.status = static_cast<unsigned int*>(addr);
    d.queried = true;
  }
  *out = &d;
  return JVP_OK;
}

// A second stream of the current device for work that may run beside the
// caller's stream (joined back to it by an event before the call returns).
jvp_status_t side_stream(DeviceInfo* d, cudaStream_t* out) {
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!d->side) {
    cudaError_t e = cudaStreamCreateWithFlags(&d->side, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      d->side = nullptr;
      return fail(JVP_ERR_CUDA, std::string("cudaStreamCreate: ") + cudaGetErrorString(e));
    }
  }
  *out = d->side;
  return JVP_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 4-D tiled map over a [B, H, N, D] tensor with a {64, rows} box and the
// 128-byte swizzle the MMA descriptors expect (for D < 64 the box reaches past
// the row: loads fill those columns with zeros, stores skip them).  Returns
// false if the layout cannot be described (the caller then takes the
// CUDA-core path).
bool encode_map(CUtensorMap* map, int dt, const void* ptr, int64_t B, int64_t H, int64_t N,
                int64_t D, const jvp_strides_t& st, int rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int64_t e = static_cast<int64_t>(elem_size(dt));
  // A size-1 dimension's stride is never used; give it a well-formed value.
  int64_t sn = st.n, sh = st.h, sb = st.b;
  if (N == 1) sn = D;
  if (H == 1) sh = sn * N;
  if (B == 1) sb = sh * H;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sn * e), static_cast<cuuint64_t>(sh * e),
                           static_cast<cuuint64_t>(sb * e)};
  for (auto s : strides)
    if (s == 0 || s % 16 != 0 || s >= (1ull << 40)) return false;
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty =
      dt == JVP_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, ty, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D tiled map over an additive fp32 mask [Bm, Hm, Nq, Nk] (Bm, Hm = 1 where
// it broadcasts) with {32, 128} boxes and the 128-byte swizzle: one box is a
// softmax warpgroup's half of a [128 x 64] score tile.  Keys must be
// contiguous, and rows must not broadcast (each of the 128 rows is read).
bool encode_mask_map(CUtensorMap* map, const void* ptr, int64_t B, int64_t H, int64_t Nq,
                     int64_t Nk, int64_t msb, int64_t msh, int64_t msq, int64_t msk) {
  auto enc = tensor_map_encoder();
  if (!enc || msk != 1 || msq <= 0 || reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
  const int64_t Hm = msh ? H : 1, Bm = msb ? B : 1;
  // A size-1 dimension's stride is never used; give it a well-formed value.
  if (Nq == 1) msq = (Nk + 3) / 4 * 4;
  const int64_t sh = Hm > 1 ? msh : msq * Nq;
  const int64_t sb = Bm > 1 ? msb : sh * Hm;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(Nk), static_cast<cuuint64_t>(Nq),
                        static_cast<cuuint64_t>(Hm), static_cast<cuuint64_t>(Bm)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(msq * 4), static_cast<cuuint64_t>(sh * 4),
                           static_cast<cuuint64_t>(sb * 4)};
  for (auto s : strides)
    if (s == 0 || s % 16 != 0 || s >= (1ull << 40)) return false;
  cuuint32_t box[4] = {32, static_cast<cuuint32_t>(kTcBlockM), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Head dimensions the tensor-core kernels take (the D = 64 or 128 kernel,
// columns past D zero-filled by TMA): multiples of 8 (16-byte rows) up to 128.
bool tc_head_dim(int64_t D) { return D >= 8 && D <= 128 && D % 8 == 0; }

bool strides_aligned16(const jvp_strides_t& s, size_t e) {
  return (s.b * static_cast<int64_t>(e)) % 16 == 0 && (s.h * static_cast<int64_t>(e)) % 16 == 0 &&
         (s.n * static_cast<int64_t>(e)) % 16 == 0;
}

Strides to_strides(const jvp_strides_t& s) { return Strides{s.b, s.h, s.n}; }

// Key/value head count (0 = H) and its check: H must be a multiple of it.
jvp_status_t kv_heads(const jvp_shape_t* shape, int64_t* hkv) {
  const int64_t H = shape->H;
  *hkv = shape->Hkv == 0 ? H : shape->Hkv;
  if (shape->Hkv < 0) return fail(JVP_ERR_INVALID_ARG, "negative Hkv");
  if (H > 0 && H % *hkv != 0)
    return fail(JVP_ERR_INVALID_ARG, "H must be a multiple of Hkv (grouped-query attention)");
  return JVP_OK;
}

// Mask kind as the kernels see it: the combined kinds become a bool or
// additive mask plus the causal flag.
void split_mask_kind(int kind, int* base, int* causal) {
  *causal = (kind == JVP_MASK_BOOL_CAUSAL || kind == JVP_MASK_ADDITIVE_CAUSAL) ? 1 : 0;
  *base = kind == JVP_MASK_BOOL_CAUSAL ? JVP_MASK_BOOL
          : kind == JVP_MASK_ADDITIVE_CAUSAL ? JVP_MASK_ADDITIVE
                                             : kind;
}

// Split-KV heuristic of the tensor-core forward: split the key range only
// when the query tiles alone would keep at most half of the SMs busy, into at
// most 16 ranges of at least 16 key tiles (1024 keys) each.  Shorter ranges
// do not pay: a CTA's fixed cost (Q load, TMEM set-up, epilogue) and the merge
// kernel then outweigh the shorter loop (measured at N = 512 and 1024 with
// B*H = 16: split runs were slower).
int choose_splits(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int num_sms) {
  const int64_t base = ((Nq + kTcBlockM - 1) / kTcBlockM) * B * H;
  if (base <= 0 || 2 * base > num_sms) return 1;
  const int64_t by_sms = (num_sms + base - 1) / base;
  const int64_t by_keys = ((Nk + kTcBlockN - 1) / kTcBlockN) / 16;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({by_sms, by_keys, 16})));
}

// Key-range split between the two CTAs of a cluster (D <= 64, fused forward +
// JVP): for problems whose query tiles fill at most half of the SMs, each
// tile's key loop is shared by two CTAs and rank 1's partial state is merged
// into rank 0's epilogue through distributed shared memory (no workspace, no
// second launch).  The hand-over of rank 1's 70 KB state takes ~4400 cycles
// and the doubled grid slows every CTA's first loads, which halving the loop
// repays from 16 key tiles on (measured: B=1 H=8 N=1024 22.5 -> 20.5 us,
// B=1 H=4 N=2048 causal 34.8 -> 26.6 us; at 8 key tiles, B=2 H=8 N=512,
// 16.4 us single pass against 18.4 us split).
bool choose_cluster_split(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int num_sms) {
  const int64_t ctas = ((Nq + kTcBlockM - 1) / kTcBlockM) * B * H;
  const int64_t key_tiles = (Nk + kTcBlockN - 1) / kTcBlockN;
  return ctas > 0 && 2 * ctas <= num_sms && key_tiles >= 16;
}

// Shared body of jvp_attn_fwd_dual(_ws) and jvp_attn_fwd.
jvp_status_t forward(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* const* in,
                     const jvp_strides_t* in_strides, const jvp_mask_t* mask, float scale,
                     void* const* out, const jvp_strides_t* out_strides, float* lse, float* mu,
                     void* stream_ptr, bool tangent, void* workspace = nullptr,
                     size_t ws_bytes = 0) {
  t_last_path = 0;
  const int n_in = tangent ? 6 : 3, n_out = tangent ? 2 : 1;
  if (!shape) return fail(JVP_ERR_INVALID_ARG, "shape is NULL");
  const int64_t B = shape->B, H = shape->H, Nq = shape->Nq, Nk = shape->Nk, D = shape->D;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return fail(JVP_ERR_INVALID_ARG, "negative size");
  if (D <= 0) return fail(JVP_ERR_INVALID_ARG, "D must be positive");
  if (D > 128) return fail(JVP_ERR_UNSUPPORTED, "D > 128 is not supported");
  if (dtype != JVP_F32 && dtype != JVP_F16 && dtype != JVP_BF16)
    return fail(JVP_ERR_INVALID_ARG, "unknown dtype");
  if (!in_strides || !out_strides) return fail(JVP_ERR_INVALID_ARG, "strides are NULL");
  if (!std::isfinite(scale)) return fail(JVP_ERR_INVALID_ARG, "scale is not finite");
  if (!dims_in_range(shape)) return fail(JVP_ERR_UNSUPPORTED, "a size exceeds 2^31 - 1");
  int64_t bh = 0, q_tiles = 0, q_groups = 0;
  if (!checked_product({B, H}, &bh) || bh > kMaxDim ||
      !checked_product({(Nq + 127) / 128, bh}, &q_tiles) || q_tiles > kMaxDim ||
      !checked_product({(Nq + 7) / 8, bh}, &q_groups) || q_groups > kMaxDim)
    return fail(JVP_ERR_UNSUPPORTED, "problem too large for one launch");
  for (int t = 0; t < n_in; ++t) {
    const jvp_strides_t& s = in_strides[t];
    if (s.d != 1) return fail(JVP_ERR_INVALID_ARG, "innermost (d) stride must be 1");
    if (s.b < 0 || s.h < 0 || s.n < 0) return fail(JVP_ERR_INVALID_ARG, "negative stride");
  }
  for (int t = 0; t < n_out; ++t) {
    const jvp_strides_t& s = out_strides[t];
    if (s.d != 1) return fail(JVP_ERR_INVALID_ARG, "innermost (d) stride of an output must be 1");
    if (s.b < 0 || s.h < 0 || s.n < 0) return fail(JVP_ERR_INVALID_ARG, "negative stride");
  }
  int64_t Hkv = 0;
  if (kv_heads(shape, &Hkv) != JVP_OK) return JVP_ERR_INVALID_ARG;
  int kind = JVP_MASK_NONE, causal_flag = 0;
  const void* mptr = nullptr;
  int64_t msb = 0, msh = 0, msq = 0, msk = 0;
  if (mask) {
    mptr = mask->ptr;
    msb = mask->stride_b, msh = mask->stride_h, msq = mask->stride_q, msk = mask->stride_k;
    if (mask->kind < JVP_MASK_NONE || mask->kind > JVP_MASK_ADDITIVE_CAUSAL)
      return fail(JVP_ERR_INVALID_ARG, "unknown mask kind");
    split_mask_kind(mask->kind, &kind, &causal_flag);
    if (kind == JVP_MASK_CAUSAL && mptr)
      return fail(JVP_ERR_INVALID_ARG,
                  "JVP_MASK_CAUSAL takes no mask tensor (use JVP_MASK_BOOL_CAUSAL or "
                  "JVP_MASK_ADDITIVE_CAUSAL)");
    if (kind == JVP_MASK_NONE && mptr)
      return fail(JVP_ERR_INVALID_ARG, "mask kind NONE with a mask tensor");
    if ((kind == JVP_MASK_BOOL || kind == JVP_MASK_ADDITIVE) && !mptr && bh > 0 && Nq > 0 &&
        Nk > 0)
      return fail(JVP_ERR_INVALID_ARG, "mask tensor is NULL");
    if (msb < 0 || msh < 0 || msq < 0 || msk < 0) return fail(JVP_ERR_INVALID_ARG, "negative mask stride");
    if (kind == JVP_MASK_ADDITIVE && !aligned(mptr, 4))
      return fail(JVP_ERR_ALIGNMENT, "additive mask is not 4-byte aligned");
  }
  const size_t e = elem_size(dtype);
  const bool rows_exist = bh > 0 && Nq > 0;
  if (!rows_exist) {
    t_last_path = 0;
    return ok();  // nothing to compute
  }
  for (int t = 0; t < n_in; ++t) {
    const bool is_q = (t == 0 || t == 3);
    if (!in[t] && (is_q || Nk > 0)) return fail(JVP_ERR_INVALID_ARG, "input pointer is NULL");
    if (!aligned(in[t], e)) return fail(JVP_ERR_ALIGNMENT, "input not aligned to its element size");
  }
  for (int t = 0; t < n_out; ++t) {
    if (!out[t]) return fail(JVP_ERR_INVALID_ARG, "output pointer is NULL");
    if (!aligned(out[t], e)) return fail(JVP_ERR_ALIGNMENT, "output not aligned to its element size");
  }
  if (!aligned(lse, 4) || !aligned(mu, 4)) return fail(JVP_ERR_ALIGNMENT, "lse/mu not 4-byte aligned");
  if (workspace && !aligned(workspace, 16))
    return fail(JVP_ERR_ALIGNMENT, "workspace is not 16-byte aligned");

  DeviceInfo* dev = nullptr;
  jvp_status_t s = current_device(&dev);
  if (s != JVP_OK) return s;
  if (!dev->sm103)
    return fail(JVP_ERR_UNSUPPORTED, "the current device is not an sm_103 (GB300-class) GPU");

  FwdParams p{};
  p.splits = 1;
  p.split_ws = nullptr;
  p.B = static_cast<int>(B);
  p.H = static_cast<int>(H);
  p.Nq = static_cast<int>(Nq);
  p.Nk = static_cast<int>(Nk);
  p.D = static_cast<int>(D);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask = mptr;
  p.msb = msb, p.msh = msh, p.msq = msq, p.msk = msk;
  p.causal = causal_flag;
  p.kv_group = static_cast<int>(H / Hkv);
  const size_t me = (kind == JVP_MASK_ADDITIVE) ? 4 : 1;
  p.mask_vec = (mptr && msk == 1 && aligned(mptr, 16) && (msq * me) % 16 == 0 &&
                (msh * me) % 16 == 0 && (msb * me) % 16 == 0)
                   ? 1
                   : 0;
  p.q = in[0], p.k = in[1], p.v = in[2];
  p.sq = to_strides(in_strides[0]), p.sk = to_strides(in_strides[1]), p.sv = to_strides(in_strides[2]);
  if (tangent) {
    p.dq = in[3], p.dk = in[4], p.dv = in[5];
    p.sdq = to_strides(in_strides[3]), p.sdk = to_strides(in_strides[4]),
    p.sdv = to_strides(in_strides[5]);
    p.t_o = out[1];
    p.sto = to_strides(out_strides[1]);
  }
  p.o = out[0];
  p.so = to_strides(out_strides[0]);
  p.lse = lse;
  p.mu = tangent ? mu : nullptr;
  p.status = dev->status;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  // Tensor-core path: fp16/bf16, D a multiple of 8 up to 128, a nonzero
  // scale, at least one key, and every tensor 16-byte aligned with
  // 16-byte-multiple strides.  D <= 64 runs the D = 64 kernel and larger D the
  // D = 128 kernel: the tensor maps' 64-column boxes reach past the D columns
  // of each row, TMA fills those with zeros (they add nothing to Q K^T,
  // dQ K^T or Q dK^T and give zero columns of A and T), and the output maps'
  // stores drop them.
  bool tc = (dtype == JVP_F16 || dtype == JVP_BF16) && tc_head_dim(D) && scale != 0.f && Nk > 0;
  const int kernel_d = D <= 64 ? 64 : 128;
  for (int t = 0; tc && t < n_in; ++t)
    tc = aligned(in[t], 16) && strides_aligned16(in_strides[t], e);
  for (int t = 0; tc && t < n_out; ++t)
    tc = aligned(out[t], 16) && strides_aligned16(out_strides[t], e);
  if (tc && scale < 0.f) {  // negated score products, |scale| (see FwdParams)
    p.neg_scores = 1;
    p.scale = -scale;
    p.scale_log2 = -scale * 1.4426950408889634f;
  }
  TcMaps maps;
  if (tc) {
    const int64_t Ns[6] = {Nq, Nk, Nk, Nq, Nk, Nk};
    CUtensorMap* dst[6] = {&maps.q, &maps.k, &maps.v, &maps.dq, &maps.dk, &maps.dv};
    for (int t = 0; tc && t < n_in; ++t) {
      const bool on_q = (t == 0 || t == 3);
      tc = encode_map(dst[t], dtype, in[t], B, on_q ? H : Hkv, Ns[t], D, in_strides[t],
                      on_q ? kTcBlockM : kTcBlockN);
    }
    if (tc && !tangent) {
      maps.dq = maps.q, maps.dk = maps.k, maps.dv = maps.v;
    }
    if (tc) tc = encode_map(&maps.o, dtype, out[0], B, H, Nq, D, out_strides[0], kTcBlockM);
    if (tc && tangent)
      tc = encode_map(&maps.t_o, dtype, out[1], B, H, Nq, D, out_strides[1], kTcBlockM);
    if (tc && !tangent) maps.t_o = maps.o;
    // The additive mask at D = 128 through shared memory (else per-row loads).
    if (tc && kind == JVP_MASK_ADDITIVE && kernel_d == 128)
      p.mask_tma = encode_mask_map(&maps.msk, mptr, B, H, Nq, Nk, msb, msh, msq, msk) ? 1 : 0;
  }
  cudaError_t err;
  if (tc) {
    p.num_q_tiles = static_cast<int>((Nq + kTcBlockM - 1) / kTcBlockM);
    // About one wave of CTAs per group of heads (one CTA per SM).
    p.group_heads = std::max(1, std::min(static_cast<int>(B * H), dev->num_sms / p.num_q_tiles));
    // Causal: the query tiles of a group run longest first, so a launch ends
    // on short tiles only within its last group.  Larger groups, as many heads
    // as keep their key/value tiles within 32 MB of L2, shorten the tail
    // (measured: 2-6 % at N = 1024..8192, D = 64 and 128).
    if (kind == JVP_MASK_CAUSAL || causal_flag) {
      const double kv_head = (tangent ? 4.0 : 2.0) * static_cast<double>(Nk) * D * e;
      const int g_l2 = static_cast<int>((32.0 * 1048576.0) / kv_head);
      p.group_heads = std::max(p.group_heads, std::min(static_cast<int>(B * H), g_l2));
    }
    // Split-KV when the caller gave a large enough workspace and it pays (its
    // partial states are laid out for the kernel's D, so D < 64 does not split).
    const int splits = (D == kernel_d) ? choose_splits(B, H, Nq, Nk, dev->num_sms) : 1;
    if (tangent && workspace && splits > 1 &&
        ws_bytes >= SplitLayout::bytes(B * H * Nq, static_cast<int>(D), splits)) {
      p.splits = splits;
      p.split_ws = static_cast<float*>(workspace);
    } else if (tangent && kernel_d == 64 && g_cluster_split.load(std::memory_order_relaxed) &&
               choose_cluster_split(B, H, Nq, Nk, dev->num_sms)) {
      p.splits = 2;  // with split_ws == nullptr: the cluster split
    }
    err = launch_fwd_tc(static_cast<DType>(dtype), kernel_d, kind, tangent, maps, p, stream);
    if (err == cudaSuccess && p.splits > 1 && p.split_ws)
      err = launch_fwd_combine(static_cast<DType>(dtype), tangent, p, stream);
    t_last_path = p.splits > 1 ? (p.split_ws ? 3 : 4) : 1;
  } else {
    p.num_q_tiles = static_cast<int>((Nq + 7) / 8);
    err = launch_fwd_simt(static_cast<DType>(dtype), kind, tangent, p, stream);
    t_last_path = 2;
  }
  if (err != cudaSuccess)
    return fail(JVP_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(err));
  return ok();
}

// Body of jvp_attn_bwd_dual and (primal = true: the tangent inputs dq, dk,
// dv, t_o, g_to, mu and outputs g_dq, g_dk, g_dv are absent) jvp_attn_bwd.
// fork: the key-side tensor-core kernels run on a second stream beside the
// query-side one (the two write disjoint gradients), joined back by an event.
jvp_status_t backward(bool primal, const jvp_shape_t* shape, jvp_dtype_t dtype,
                      const void* const* in, const float* lse, const float* mu,
                      const jvp_strides_t* in_strides, const jvp_mask_t* mask, float scale,
                      void* const* out, const jvp_strides_t* out_strides, void* workspace,
                      size_t ws_bytes, void* stream_ptr, bool fork = true) {
  t_last_path = 0;
  if (!shape) return fail(JVP_ERR_INVALID_ARG, "shape is NULL");
  const int64_t B = shape->B, H = shape->H, Nq = shape->Nq, Nk = shape->Nk, D = shape->D;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return fail(JVP_ERR_INVALID_ARG, "negative size");
  if (D <= 0) return fail(JVP_ERR_INVALID_ARG, "D must be positive");
  if (D > 128) return fail(JVP_ERR_UNSUPPORTED, "D > 128 is not supported");
  if (dtype != JVP_F32 && dtype != JVP_F16 && dtype != JVP_BF16)
    return fail(JVP_ERR_INVALID_ARG, "unknown dtype");
  if (!in_strides || !out_strides) return fail(JVP_ERR_INVALID_ARG, "strides are NULL");
  if (!std::isfinite(scale)) return fail(JVP_ERR_INVALID_ARG, "scale is not finite");
  if (!dims_in_range(shape)) return fail(JVP_ERR_UNSUPPORTED, "a size exceeds 2^31 - 1");
  int64_t bh = 0, q_rows = 0, k_rows = 0;
  if (!checked_product({B, H}, &bh) || !checked_product({bh, Nq}, &q_rows) ||
      q_rows > kMaxDim / 32 || !checked_product({bh, Nk}, &k_rows) || k_rows > kMaxDim)
    return fail(JVP_ERR_UNSUPPORTED, "problem too large for one launch");
  for (int t = 0; t < 10; ++t) {
    const jvp_strides_t& s = in_strides[t];
    if (s.d != 1) return fail(JVP_ERR_INVALID_ARG, "innermost (d) stride must be 1");
    if (s.b < 0 || s.h < 0 || s.n < 0) return fail(JVP_ERR_INVALID_ARG, "negative stride");
  }
  for (int t = 0; t < 6; ++t) {
    const jvp_strides_t& s = out_strides[t];
    if (s.d != 1) return fail(JVP_ERR_INVALID_ARG, "innermost (d) stride of an output must be 1");
    if (s.b < 0 || s.h < 0 || s.n < 0) return fail(JVP_ERR_INVALID_ARG, "negative stride");
  }
  int64_t Hkv = 0;
  if (kv_heads(shape, &Hkv) != JVP_OK) return JVP_ERR_INVALID_ARG;
  int kind = JVP_MASK_NONE, causal_flag = 0;
  const void* mptr = nullptr;
  int64_t msb = 0, msh = 0, msq = 0, msk = 0;
  if (mask) {
    mptr = mask->ptr;
    msb = mask->stride_b, msh = mask->stride_h, msq = mask->stride_q, msk = mask->stride_k;
    if (mask->kind < JVP_MASK_NONE || mask->kind > JVP_MASK_ADDITIVE_CAUSAL)
      return fail(JVP_ERR_INVALID_ARG, "unknown mask kind");
    split_mask_kind(mask->kind, &kind, &causal_flag);
    if ((kind == JVP_MASK_CAUSAL || kind == JVP_MASK_NONE) && mptr)
      return fail(JVP_ERR_INVALID_ARG, "this mask kind takes no mask tensor");
    if ((kind == JVP_MASK_BOOL || kind == JVP_MASK_ADDITIVE) && !mptr && q_rows > 0 && Nk > 0)
      return fail(JVP_ERR_INVALID_ARG, "mask tensor is NULL");
    if (msb < 0 || msh < 0 || msq < 0 || msk < 0) return fail(JVP_ERR_INVALID_ARG, "negative mask stride");
    if (kind == JVP_MASK_ADDITIVE && !aligned(mptr, 4))
      return fail(JVP_ERR_ALIGNMENT, "additive mask is not 4-byte aligned");
  }
  if (q_rows == 0 && k_rows == 0) return ok();  // nothing to compute
  const size_t e = elem_size(dtype);
  // tangent-side entries: inputs dq dk dv t_o g_to, outputs g_dq g_dk g_dv
  auto tangent_in = [](int t) { return t == 3 || t == 4 || t == 5 || t == 7 || t == 9; };
  for (int t = 0; t < 10; ++t) {
    if (primal && tangent_in(t)) continue;
    const bool on_keys = (t == 1 || t == 2 || t == 4 || t == 5);
    if (!in[t] && (!on_keys || Nk > 0) && (on_keys || Nq > 0))
      return fail(JVP_ERR_INVALID_ARG, "input pointer is NULL");
    if (!aligned(in[t], e)) return fail(JVP_ERR_ALIGNMENT, "input not aligned to its element size");
  }
  for (int t = 0; t < (primal ? 3 : 6); ++t) {
    const bool on_keys = (t == 1 || t == 2 || t == 4 || t == 5);
    if (!out[t] && (!on_keys || Nk > 0) && (on_keys || Nq > 0))
      return fail(JVP_ERR_INVALID_ARG, "output pointer is NULL");
    if (!aligned(out[t], e)) return fail(JVP_ERR_ALIGNMENT, "output not aligned to its element size");
  }
  if (Nq > 0 && !lse) return fail(JVP_ERR_INVALID_ARG, "lse is required");
  if (Nq > 0 && !primal && !mu) return fail(JVP_ERR_INVALID_ARG, "lse and mu are required");
  if (!aligned(lse, 4) || !aligned(mu, 4)) return fail(JVP_ERR_ALIGNMENT, "lse/mu not 4-byte aligned");
  const size_t need = bwd_workspace_bytes(q_rows);
  if (need > 0 && (!workspace || ws_bytes < need))
    return fail(JVP_ERR_WORKSPACE, "workspace is NULL or smaller than jvp_attn_bwd_dual_workspace_size()");
  if (!aligned(workspace, 4)) return fail(JVP_ERR_ALIGNMENT, "workspace is not 4-byte aligned");

  DeviceInfo* dev = nullptr;
  jvp_status_t s = current_device(&dev);
  if (s != JVP_OK) return s;
  if (!dev->sm103)
    return fail(JVP_ERR_UNSUPPORTED, "the current device is not an sm_103 (GB300-class) GPU");

  BwdParams p{};
  p.B = static_cast<int>(B), p.H = static_cast<int>(H), p.Nq = static_cast<int>(Nq);
  p.Nk = static_cast<int>(Nk), p.D = static_cast<int>(D);
  p.scale = scale;
  p.mask_kind = kind;
  p.causal = causal_flag;
  p.kv_group = static_cast<int>(H / Hkv);
  p.mask = mptr;
  p.msb = msb, p.msh = msh, p.msq = msq, p.msk = msk;
  {
    const int64_t me = (kind == JVP_MASK_ADDITIVE) ? 4 : 1;
    p.mask_vec = (mptr && msk == 1 && aligned(mptr, 16) && (msq * me) % 16 == 0 &&
                  (msh * me) % 16 == 0 && (msb * me) % 16 == 0)
                     ? 1
                     : 0;
  }
  p.q = in[0], p.k = in[1], p.v = in[2], p.dq = in[3], p.dk = in[4], p.dv = in[5];
  p.o = in[6], p.t_o = in[7], p.g_o = in[8], p.g_to = in[9];
  Strides* sin[10] = {&p.sq, &p.sk, &p.sv, &p.sdq, &p.sdk, &p.sdv, &p.so, &p.sto, &p.sgo, &p.sgto};
  for (int t = 0; t < 10; ++t) *sin[t] = to_strides(in_strides[t]);
  p.lse = lse, p.mu = mu;
  p.g_q = out[0], p.g_k = out[1], p.g_v = out[2], p.g_dq = out[3], p.g_dk = out[4], p.g_dv = out[5];
  Strides* sout[6] = {&p.sgq, &p.sgk, &p.sgv, &p.sgdq, &p.sgdk, &p.sgdv};
  for (int t = 0; t < 6; ++t) *sout[t] = to_strides(out_strides[t]);
  p.nu = static_cast<float*>(workspace);
  p.delta = p.nu + q_rows;
  p.primal = primal ? 1 : 0;
  p.ksplits = 1;
  p.kws = nullptr;
  p.qsplits = 1;
  p.qws = nullptr;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  // Tensor-core path: fp16/bf16, D in {16, 32, 64, 128}, at least one row and
  // one key, every tensor 16-byte aligned with 16-byte-multiple strides.  As in
  // the forward, D = 16 and 32 run the D = 64 kernels on zero-filled columns
  // (their gradient stores stop at D).
  bool tc = (dtype == JVP_F16 || dtype == JVP_BF16) && tc_head_dim(D) && Nq > 0 && Nk > 0;
  for (int t = 0; tc && t < 10; ++t) tc = aligned(in[t], 16) && strides_aligned16(in_strides[t], e);
  for (int t = 0; tc && t < 6; ++t) tc = aligned(out[t], 16) && strides_aligned16(out_strides[t], e);
  // Tensor maps: qm for the query-major kernel (query side 128 rows, key side
  // 64); km for the key-major kernel (key side 128 rows, query side 32, and 64
  // for its value part at D = 128).
  BwdTcMaps qm, km;
  if (tc) {
    // in order: q k v dq dk dv o t_o g_o g_to
    const int64_t Ns[10] = {Nq, Nk, Nk, Nq, Nk, Nk, Nq, Nq, Nq, Nq};
    const int qidx[4] = {0, 3, 8, 9}, kidx[4] = {1, 4, 2, 5};
    CUtensorMap* qdst_q[4] = {&qm.q, &qm.dq, &qm.go, &qm.gto};
    CUtensorMap* qdst_k[4] = {&qm.k, &qm.dk, &qm.v, &qm.dv};
    CUtensorMap* kdst_q[4] = {&km.q, &km.dq, &km.go, &km.gto};
    CUtensorMap* kdst_q64[4] = {&km.q64, &km.dq64, &km.go64, &km.gto64};
    CUtensorMap* kdst_k[4] = {&km.k, &km.dk, &km.v, &km.dv};
    for (int u = 0; tc && u < 4; ++u) {
      if (primal && (u == 1 || u == 3)) continue;  // dq/dk and g_to/dv: absent
      const int a = qidx[u], c = kidx[u];
      tc = encode_map(qdst_q[u], dtype, in[a], B, H, Ns[a], D, in_strides[a], 128) &&
           encode_map(qdst_k[u], dtype, in[c], B, Hkv, Ns[c], D, in_strides[c], 64) &&
           encode_map(kdst_q[u], dtype, in[a], B, H, Ns[a], D, in_strides[a], 32) &&
           encode_map(kdst_q64[u], dtype, in[a], B, H, Ns[a], D, in_strides[a], 64) &&
           encode_map(kdst_k[u], dtype, in[c], B, Hkv, Ns[c], D, in_strides[c], 128);
    }
  }
  cudaError_t err;
  if (tc) {
    // Few key-major CTAs (grouped-query heads, small B * Hkv): split each key
    // tile's query tiles over several CTAs when the workspace has room for
    // their partial sums.
    // The same for few query-major CTAs walking many key tiles (few queries,
    // many keys): each query tile's key tiles over several CTAs.
    const int kd = D <= 64 ? 64 : 128;
    const int ks = bwd_key_splits(B, Hkv, Nq, Nk, H / Hkv, dev->num_sms);
    const int qs = bwd_query_splits(B, H, Nq, Nk, dev->num_sms);
    const size_t base = (bwd_workspace_bytes(q_rows) + 255) & ~static_cast<size_t>(255);
    const size_t kbytes = bwd_key_split_bytes(ks, B, Hkv, Nk, kd);
    const size_t qbytes = bwd_query_split_bytes(qs, B, H, Nq, kd);
    // (The no-allocation entry point, `fork` false, keeps its fixed scratch
    // for nu and delta and runs unsplit.)
    if (fork && aligned(workspace, 16) && ws_bytes >= base + kbytes + qbytes) {
      if (ks > 1) {
        p.ksplits = ks;
        p.kws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + base);
      }
      if (qs > 1) {
        p.qsplits = qs;
        p.qws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + base + kbytes);
      }
    }
    err = launch_bwd_rows(static_cast<DType>(dtype), p, stream);
    // After the row pass the query-major and key-major kernels are
    // independent: the key side goes to the side stream, so the CTAs of
    // either fill the SMs the other's last wave leaves idle.
    cudaStream_t kstream = stream;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    if (err == cudaSuccess && fork) {
      cudaStream_t side = nullptr;
      if (side_stream(dev, &side) == JVP_OK &&
          cudaEventCreateWithFlags(&ev_fork, cudaEventDisableTiming) == cudaSuccess &&
          cudaEventCreateWithFlags(&ev_join, cudaEventDisableTiming) == cudaSuccess &&
          cudaEventRecord(ev_fork, stream) == cudaSuccess &&
          cudaStreamWaitEvent(side, ev_fork, 0) == cudaSuccess) {
        kstream = side;
      }
    }
    if (err == cudaSuccess)
      err = launch_bwd_tc(static_cast<DType>(dtype), D <= 64 ? 64 : 128, kind, primal, qm, km, p,
                          dev->num_sms, dev->status, stream, kstream);
    if (kstream != stream) {  // join (also after a failed launch)
      cudaError_t ej = cudaEventRecord(ev_join, kstream);
      if (ej == cudaSuccess) ej = cudaStreamWaitEvent(stream, ev_join, 0);
      if (err == cudaSuccess) err = ej;
    }
    if (ev_fork) cudaEventDestroy(ev_fork);  // (released once the recorded work completes)
    if (ev_join) cudaEventDestroy(ev_join);
    t_last_path = 1;
  } else {
    err = launch_bwd_simt(static_cast<DType>(dtype), p, stream);
    t_last_path = 2;
  }
  if (err != cudaSuccess)
    return fail(JVP_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(err));
  return ok();
}

__global__ void wait_timeout_selftest_kernel(long long limit, unsigned int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_barrier_init();
  // Nothing ever arrives on `bar`: the bounded wait must give up.
  if (!mbar_wait(&bar, 0, &abort_flag, limit)) atomicOr(status, 1u);
}

}  // namespace

cudaError_t launch_fwd_tc(DType dt, int D, int mask_kind, bool tangent, const TcMaps& maps,
                          const FwdParams& p, cudaStream_t stream) {
  if (dt == kF16 && D == 64) return launch_fwd_tc_f16_d64(mask_kind, tangent, maps, p, stream);
  if (dt == kF16 && D == 128) return launch_fwd_tc_f16_d128(mask_kind, tangent, maps, p, stream);
  if (dt == kBF16 && D == 64) return launch_fwd_tc_bf16_d64(mask_kind, tangent, maps, p, stream);
  if (dt == kBF16 && D == 128) return launch_fwd_tc_bf16_d128(mask_kind, tangent, maps, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_tc(DType dt, int D, int mask_kind, bool primal, const BwdTcMaps& qmaps,
                          const BwdTcMaps& kmaps, const BwdParams& p, int num_sms,
                          unsigned int* status, cudaStream_t stream, cudaStream_t kstream) {
#define JVP_BWD_CALL(NAME) NAME(mask_kind, qmaps, kmaps, p, num_sms, status, stream, kstream)
  if (primal) {
    if (dt == kF16 && D == 64) return JVP_BWD_CALL(launch_bwd_primal_tc_f16_d64);
    if (dt == kF16 && D == 128) return JVP_BWD_CALL(launch_bwd_primal_tc_f16_d128);
    if (dt == kBF16 && D == 64) return JVP_BWD_CALL(launch_bwd_primal_tc_bf16_d64);
    if (dt == kBF16 && D == 128) return JVP_BWD_CALL(launch_bwd_primal_tc_bf16_d128);
    return cudaErrorInvalidValue;
  }
  if (dt == kF16 && D == 64) return JVP_BWD_CALL(launch_bwd_tc_f16_d64);
  if (dt == kF16 && D == 128) return JVP_BWD_CALL(launch_bwd_tc_f16_d128);
  if (dt == kBF16 && D == 64) return JVP_BWD_CALL(launch_bwd_tc_bf16_d64);
  if (dt == kBF16 && D == 128) return JVP_BWD_CALL(launch_bwd_tc_bf16_d128);
#undef JVP_BWD_CALL
  return cudaErrorInvalidValue;
}

}  // namespace jvp

extern "C" {

jvp_status_t jvp_attn_fwd_dual(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                               const void* k, const void* v, const void* dq, const void* dk,
                               const void* dv, const jvp_strides_t* in_strides,
                               const jvp_mask_t* mask, float scale, void* o, void* t_o,
                               const jvp_strides_t* out_strides, float* lse, float* mu,
                               void* stream) {
  const void* in[6] = {q, k, v, dq, dk, dv};
  void* out[2] = {o, t_o};
  return jvp::forward(shape, dtype, in, in_strides, mask, scale, out, out_strides, lse, mu, stream,
                      true);
}

jvp_status_t jvp_attn_fwd_dual_ws(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                                  const void* k, const void* v, const void* dq, const void* dk,
                                  const void* dv, const jvp_strides_t* in_strides,
                                  const jvp_mask_t* mask, float scale, void* o, void* t_o,
                                  const jvp_strides_t* out_strides, float* lse, float* mu,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const void* in[6] = {q, k, v, dq, dk, dv};
  void* out[2] = {o, t_o};
  return jvp::forward(shape, dtype, in, in_strides, mask, scale, out, out_strides, lse, mu, stream,
                      true, workspace, workspace_bytes);
}

size_t jvp_attn_fwd_dual_workspace_size(const jvp_shape_t* shape, jvp_dtype_t dtype) {
  if (!shape || shape->B <= 0 || shape->H <= 0 || shape->Nq <= 0 || shape->Nk <= 0) return 0;
  int64_t rows = 0;
  if (!jvp::dims_in_range(shape) || !jvp::checked_product({shape->B, shape->H, shape->Nq}, &rows) ||
      rows > jvp::kMaxDim * 128)
    return 0;  // the call itself rejects this shape
  if ((dtype != JVP_F16 && dtype != JVP_BF16) || (shape->D != 64 && shape->D != 128)) return 0;
  jvp::DeviceInfo* dev = nullptr;
  if (jvp::current_device(&dev) != JVP_OK || !dev->sm103) {
    cudaGetLastError();  // no usable device: no split, no workspace
    return 0;
  }
  const int splits = jvp::choose_splits(shape->B, shape->H, shape->Nq, shape->Nk, dev->num_sms);
  if (splits <= 1) return 0;
  return jvp::SplitLayout::bytes(shape->B * shape->H * shape->Nq, static_cast<int>(shape->D),
                                 splits);
}

jvp_status_t jvp_attn_fwd(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                          const void* k, const void* v, const jvp_strides_t* in_strides,
                          const jvp_mask_t* mask, float scale, void* o,
                          const jvp_strides_t* out_strides, float* lse, void* stream) {
  const void* in[3] = {q, k, v};
  void* out[1] = {o};
  return jvp::forward(shape, dtype, in, in_strides, mask, scale, out, out_strides, lse, nullptr,
                      stream, false);
}

jvp_status_t jvp_attn_bwd_dual(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                               const void* k, const void* v, const void* dq, const void* dk,
                               const void* dv, const void* o, const void* t_o, const float* lse,
                               const float* mu, const void* g_o, const void* g_to,
                               const jvp_strides_t* in_strides, const jvp_mask_t* mask,
                               float scale, void* g_q, void* g_k, void* g_v, void* g_dq,
                               void* g_dk, void* g_dv, const jvp_strides_t* out_strides,
                               void* workspace, size_t workspace_bytes, void* stream) {
  const void* in[10] = {q, k, v, dq, dk, dv, o, t_o, g_o, g_to};
  void* out[6] = {g_q, g_k, g_v, g_dq, g_dk, g_dv};
  return jvp::backward(false, shape, dtype, in, lse, mu, in_strides, mask, scale, out,
                       out_strides, workspace, workspace_bytes, stream);
}

// jvp_attn_bwd_dual on one stream (no side stream, no events): the body of
// jvp_attn_bwd_dual_noalloc.
static jvp_status_t bwd_dual_one_stream(const jvp_shape_t* shape, jvp_dtype_t dtype,
                                        const void* const* in, const float* lse,
                                        const float* mu, const jvp_strides_t* in_strides,
                                        const jvp_mask_t* mask, float scale, void* const* out,
                                        const jvp_strides_t* out_strides, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  return jvp::backward(false, shape, dtype, in, lse, mu, in_strides, mask, scale, out,
                       out_strides, workspace, workspace_bytes, stream, false);
}

jvp_status_t jvp_attn_bwd(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                          const void* k, const void* v, const void* o, const float* lse,
                          const void* g_o, const jvp_strides_t* in_strides,
                          const jvp_mask_t* mask, float scale, void* g_q, void* g_k, void* g_v,
                          const jvp_strides_t* out_strides, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!in_strides || !out_strides) return jvp::fail(JVP_ERR_INVALID_ARG, "strides are NULL");
  // The dual backward's argument layout with the tangent entries absent (a
  // unit-stride placeholder record each).
  const jvp_strides_t none{0, 0, 0, 1};
  const jvp_strides_t ins[10] = {in_strides[0], in_strides[1], in_strides[2], none, none, none,
                                 in_strides[3], none, in_strides[4], none};
  const jvp_strides_t outs[6] = {out_strides[0], out_strides[1], out_strides[2], none, none, none};
  const void* in[10] = {q, k, v, nullptr, nullptr, nullptr, o, nullptr, g_o, nullptr};
  void* out[6] = {g_q, g_k, g_v, nullptr, nullptr, nullptr};
  return jvp::backward(true, shape, dtype, in, lse, nullptr, ins, mask, scale, out, outs,
                       workspace, workspace_bytes, stream);
}

size_t jvp_attn_bwd_workspace_size(const jvp_shape_t* shape, jvp_dtype_t dtype) {
  return jvp_attn_bwd_dual_workspace_size(shape, dtype);
}

namespace jvp {
// Workspace of the backward without a key-major split: nu and delta.
size_t bwd_base_workspace_size(const jvp_shape_t* shape) {
  if (!shape || shape->B < 0 || shape->H < 0 || shape->Nq < 0) return 0;
  int64_t rows = 0;
  if (!dims_in_range(shape) || !checked_product({shape->B, shape->H, shape->Nq}, &rows) ||
      rows > kMaxDim)
    return SIZE_MAX;  // beyond any launch (jvp_attn_bwd_dual rejects the shape)
  return bwd_workspace_bytes(rows);
}
}  // namespace jvp

size_t jvp_attn_bwd_dual_workspace_size(const jvp_shape_t* shape, jvp_dtype_t dtype) {
  const size_t base = jvp::bwd_base_workspace_size(shape);
  if (base == 0 || base == SIZE_MAX) return base;
  // plus the key-major split's partial sums, when the tensor-core path would
  // split this shape on the current device
  const int64_t D = shape->D, Hkv = shape->Hkv ? shape->Hkv : shape->H;
  if ((dtype != JVP_F16 && dtype != JVP_BF16) || !jvp::tc_head_dim(D) ||
      shape->Nq <= 0 || shape->Nk <= 0 || Hkv <= 0 || shape->H % Hkv != 0)
    return base;
  jvp::DeviceInfo* dev = nullptr;
  if (jvp::current_device(&dev) != JVP_OK || !dev->sm103) {
    cudaGetLastError();  // no usable device: no split
    return base;
  }
  const int ks = jvp::bwd_key_splits(shape->B, Hkv, shape->Nq, shape->Nk, shape->H / Hkv,
                                     dev->num_sms);
  const int qs = jvp::bwd_query_splits(shape->B, shape->H, shape->Nq, shape->Nk, dev->num_sms);
  if (ks <= 1 && qs <= 1) return base;
  const int kd = D <= 64 ? 64 : 128;
  return ((base + 255) & ~static_cast<size_t>(255)) +
         jvp::bwd_key_split_bytes(ks, shape->B, Hkv, shape->Nk, kd) +
         jvp::bwd_query_split_bytes(qs, shape->B, shape->H, shape->Nq, kd);
}

jvp_status_t jvp_attn_get_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return jvp::fail(JVP_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, jvp::g_device_status, sizeof(word));
  if (e != cudaSuccess)
    return jvp::fail(JVP_ERR_CUDA, std::string("reading the status word: ") + cudaGetErrorString(e));
  if (word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(jvp::g_device_status, &zero, sizeof(zero));
    if (e != cudaSuccess)
      return jvp::fail(JVP_ERR_CUDA, std::string("clearing the status word: ") + cudaGetErrorString(e));
    if (word & 2u) {
      static const char* kinds[4] = {"TMEM column", "shared-memory offset", "global row",
                                     "global column"};
      std::string what;
      for (unsigned k = 0; k < 4; ++k)
        if (word & (1u << (8 + k))) what += std::string(what.empty() ? "" : ", ") + kinds[k];
      return jvp::fail(JVP_ERR_BOUNDS, "a device-side bounds check failed (" + what + ")");
    }
    return jvp::fail(JVP_ERR_DEVICE_TIMEOUT, "a device-side wait ran out of time");
  }
  return jvp::ok();
}

const char* jvp_attn_status_string(jvp_status_t status) {
  switch (status) {
    case JVP_OK: return "ok";
    case JVP_ERR_INVALID_ARG: return "invalid argument";
    case JVP_ERR_UNSUPPORTED: return "unsupported";
    case JVP_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case JVP_ERR_CUDA: return "CUDA error";
    case JVP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case JVP_ERR_WORKSPACE: return "workspace missing or too small";
    case JVP_ERR_BOUNDS: return "device-side bounds check failed (debug build)";
  }
  return "unknown status";
}

const char* jvp_attn_last_error(void) { return jvp::t_last_error.c_str(); }

int jvp_attn_version(void) { return 200; }

int jvp_attn_debug_last_path(void) { return jvp::t_last_path; }

jvp_status_t jvp_attn_debug_set_cluster_split(int enable) {
  if (enable != 0 && enable != 1) return jvp::fail(JVP_ERR_INVALID_ARG, "enable must be 0 or 1");
  jvp::g_cluster_split.store(enable, std::memory_order_relaxed);
  return jvp::ok();
}

jvp_status_t jvp_attn_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles >= (1ll << 31))
    return jvp::fail(JVP_ERR_INVALID_ARG, "limit_cycles must be in [1, 2^31)");
  jvp::DeviceInfo* dev = nullptr;
  jvp_status_t s = jvp::current_device(&dev);
  if (s != JVP_OK) return s;
  if (!dev->sm103) return jvp::fail(JVP_ERR_UNSUPPORTED, "the current device is not sm_103");
  jvp::wait_timeout_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<long long>(limit_cycles), dev->status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return jvp::fail(JVP_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(e));
  return jvp::ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Host-buffer forward (jvp_attn_fwd_dual_host): the inputs and outputs live in
// host memory; chunks of (batch, head) pairs go through a two-slot device
// staging area with their host->device copies, the fused kernel and the
// device->host copies of the previous chunk overlapped on three streams.

namespace jvp {
namespace {
struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;  // copy streams of this device
  cudaEvent_t entry = nullptr, in_ready[2] = {}, computed[2] = {}, out_done[2] = {};
};
std::mutex g_pipe_mu;  // held for the whole enqueue of a call
HostPipe g_pipe[64];

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of one staging slot for chunks of `n` (batch, head) pairs.
struct SlotLayout {
  size_t q, k, v, dq, dk, dv, o, t_o, lse, mu, bytes;
  SlotLayout(int64_t n, int64_t Nq, int64_t Nk, int64_t D, size_t e) {
    const size_t qb = up256(static_cast<size_t>(n * Nq * D) * e);
    const size_t kb = up256(static_cast<size_t>(n * Nk * D) * e);
    const size_t sb = up256(static_cast<size_t>(n * Nq) * sizeof(float));
    q = 0, dq = qb, o = 2 * qb, t_o = 3 * qb;
    k = 4 * qb, v = k + kb, dk = v + kb, dv = dk + kb;
    lse = dv + kb, mu = lse + sb;
    bytes = mu + sb;
  }
};

// Groups of (batch, head) pairs: min(chunks, BH) of them.  Their sizes fall
// linearly (weights G, G - 1, ..., 1 on the pairs left after one per group),
// so the last group -- whose kernel and device->host copies are all that
// follows the last host->device copy -- is the smallest, while the copies of
// the first groups, which run under no kernel anyway, carry the bulk.
int64_t num_groups(int64_t BH, int chunks) {
  return std::max<int64_t>(1, std::min<int64_t>(chunks, BH));
}
// First pair of group g of G (g = G gives BH): one pair per group plus the
// weighted share of the other BH - G.
int64_t group_edge(int64_t BH, int64_t G, int64_t g) {
  const unsigned __int128 rest = static_cast<unsigned __int128>(BH - G);
  const unsigned __int128 w = static_cast<unsigned __int128>(g * G - g * (g - 1) / 2);
  const unsigned __int128 total = static_cast<unsigned __int128>(G * (G + 1) / 2);
  return g + static_cast<int64_t>(rest * w / total);
}
// Pairs in the largest group (the staging slots hold one group each): exact
// for up to 2^16 groups; beyond that the bound 2 + floor(R G / T) (group g
// holds 1 + floor(R w_{g+1} / T) - floor(R w_g / T) pairs, w_{g+1} - w_g <= G).
int64_t max_group(int64_t BH, int chunks) {
  const int64_t G = num_groups(BH, chunks);
  if (G <= (1 << 16)) {
    int64_t m = 0;
    for (int64_t g = 0; g < G; ++g)
      m = std::max(m, group_edge(BH, G, g + 1) - group_edge(BH, G, g));
    return m;
  }
  const unsigned __int128 rest = static_cast<unsigned __int128>(BH - G);
  const unsigned __int128 total = static_cast<unsigned __int128>(G * (G + 1) / 2);
  const int64_t bound = 2 + static_cast<int64_t>(rest * static_cast<unsigned __int128>(G) / total);
  return std::min(BH, bound);
}

jvp_status_t host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(JVP_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(JVP_ERR_UNSUPPORTED, "device index out of range");
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming);
    for (int u = 0; u < 2 && e == cudaSuccess; ++u) {
      e = cudaEventCreateWithFlags(&hp.in_ready[u], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.computed[u], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.out_done[u], cudaEventDisableTiming);
    }
    if (e != cudaSuccess)
      return fail(JVP_ERR_CUDA, std::string("stream/event set-up: ") + cudaGetErrorString(e));
    hp.ready = true;
  }
  *out = &hp;
  return JVP_OK;
}
}  // namespace
}  // namespace jvp

extern "C" size_t jvp_attn_fwd_dual_host_workspace_size(const jvp_shape_t* shape,
                                                        jvp_dtype_t dtype, int chunks) {
  if (!shape || shape->B <= 0 || shape->H <= 0 || shape->Nq <= 0 || shape->D <= 0 ||
      shape->Nk < 0 || chunks < 1)
    return 0;
  int64_t bh = 0, rows = 0;
  if (!jvp::dims_in_range(shape) || !jvp::checked_product({shape->B, shape->H}, &bh) ||
      !jvp::checked_product({bh, shape->Nq + shape->Nk, shape->D}, &rows) || rows > (1ll << 56))
    return 0;  // the call itself rejects this shape
  const int64_t n = jvp::max_group(bh, chunks);
  return 2 * jvp::SlotLayout(n, shape->Nq, shape->Nk, shape->D, jvp::elem_size(dtype)).bytes;
}

extern "C" jvp_status_t jvp_attn_fwd_dual_host(
    const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q, const void* k, const void* v,
    const void* dq, const void* dk, const void* dv, const jvp_mask_t* mask, float scale, void* o,
    void* t_o, float* lse, float* mu, int chunks, void* workspace, size_t workspace_bytes,
    void* stream_ptr) {
  using namespace jvp;
  t_last_path = 0;
  if (!shape) return fail(JVP_ERR_INVALID_ARG, "shape is NULL");
  const int64_t B = shape->B, H = shape->H, Nq = shape->Nq, Nk = shape->Nk, D = shape->D;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || D <= 0) return fail(JVP_ERR_INVALID_ARG, "bad sizes");
  if (D > 128) return fail(JVP_ERR_UNSUPPORTED, "D > 128 is not supported");
  int64_t bh_all = 0, q_tiles = 0;
  if (!dims_in_range(shape) || !checked_product({B, H}, &bh_all) || bh_all > kMaxDim ||
      !checked_product({(Nq + 127) / 128, bh_all}, &q_tiles) || q_tiles > kMaxDim)
    return fail(JVP_ERR_UNSUPPORTED, "problem too large for one launch");
  if (dtype != JVP_F32 && dtype != JVP_F16 && dtype != JVP_BF16)
    return fail(JVP_ERR_INVALID_ARG, "unknown dtype");
  if (!std::isfinite(scale)) return fail(JVP_ERR_INVALID_ARG, "scale is not finite");
  if (shape->Hkv != 0 && shape->Hkv != H)
    return fail(JVP_ERR_UNSUPPORTED, "the host-buffer entry point takes Hkv == H only");
  if (chunks < 1) return fail(JVP_ERR_INVALID_ARG, "chunks must be >= 1");
  if (mask && (mask->stride_b != 0 || mask->stride_h != 0) && mask->ptr)
    return fail(JVP_ERR_INVALID_ARG,
                "the host-buffer entry point needs a mask shared by every (batch, head) "
                "(stride_b = stride_h = 0)");
  if (B * H * Nq == 0) return ok();
  if (!q || !dq || !o || !t_o || (Nk > 0 && (!k || !v || !dk || !dv)))
    return fail(JVP_ERR_INVALID_ARG, "input or output pointer is NULL");
  const size_t need = jvp_attn_fwd_dual_host_workspace_size(shape, dtype, chunks);
  if (!workspace || workspace_bytes < need)
    return fail(JVP_ERR_WORKSPACE,
                "workspace is NULL or smaller than jvp_attn_fwd_dual_host_workspace_size()");
  if (!aligned(workspace, 256)) return fail(JVP_ERR_ALIGNMENT, "workspace is not 256-byte aligned");

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  jvp_status_t s = host_pipe(&hp);
  if (s != JVP_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const size_t e = elem_size(dtype);
  const int64_t BH = B * H, groups = num_groups(BH, chunks);
  const SlotLayout L(max_group(BH, chunks), Nq, Nk, D, e);
  auto cu = [&](cudaError_t err, const char* what) -> jvp_status_t {
    if (err == cudaSuccess) return JVP_OK;
    return fail(JVP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(err));
  };
  // Everything starts after the work already on `stream` (a previous call may
  // still be reading the same staging area).
  if ((s = cu(cudaEventRecord(hp->entry, stream), "cudaEventRecord")) != JVP_OK) return s;
  if ((s = cu(cudaStreamWaitEvent(hp->in, hp->entry, 0), "cudaStreamWaitEvent")) != JVP_OK) return s;
  if ((s = cu(cudaStreamWaitEvent(hp->out, hp->entry, 0), "cudaStreamWaitEvent")) != JVP_OK) return s;
  int last_path = 0;
  int last_slot = 0;
  for (int64_t c = 0; c < groups; ++c) {
    const int64_t lo = group_edge(BH, groups, c);
    const int64_t n = group_edge(BH, groups, c + 1) - lo;
    const int sl = static_cast<int>(c & 1);
    last_slot = sl;
    uint8_t* base = static_cast<uint8_t*>(workspace) + sl * L.bytes;
    const size_t qbytes = static_cast<size_t>(n * Nq * D) * e, kbytes = static_cast<size_t>(n * Nk * D) * e;
    const size_t qoff = static_cast<size_t>(lo * Nq * D) * e, koff = static_cast<size_t>(lo * Nk * D) * e;
    // host -> device (after the kernel of chunk c-2 has read this slot)
    if (c >= 2 && (s = cu(cudaStreamWaitEvent(hp->in, hp->computed[sl], 0), "cudaStreamWaitEvent")) != JVP_OK)
      return s;
    struct { size_t dst; const void* src; size_t off, bytes; } cp[6] = {
        {L.q, q, qoff, qbytes}, {L.k, k, koff, kbytes}, {L.v, v, koff, kbytes},
        {L.dq, dq, qoff, qbytes}, {L.dk, dk, koff, kbytes}, {L.dv, dv, koff, kbytes}};
    for (auto& x : cp) {
      if (x.bytes == 0) continue;
      s = cu(cudaMemcpyAsync(base + x.dst, static_cast<const uint8_t*>(x.src) + x.off, x.bytes,
                             cudaMemcpyHostToDevice, hp->in),
             "cudaMemcpyAsync (host to device)");
      if (s != JVP_OK) return s;
    }
    if ((s = cu(cudaEventRecord(hp->in_ready[sl], hp->in), "cudaEventRecord")) != JVP_OK) return s;
    // the kernel on `stream` (after chunk c-2's outputs have left this slot)
    if ((s = cu(cudaStreamWaitEvent(stream, hp->in_ready[sl], 0), "cudaStreamWaitEvent")) != JVP_OK)
      return s;
    if (c >= 2 && (s = cu(cudaStreamWaitEvent(stream, hp->out_done[sl], 0), "cudaStreamWaitEvent")) != JVP_OK)
      return s;
    const jvp_shape_t cs{1, n, Nq, Nk, D, 0};
    const jvp_strides_t sq{n * Nq * D, Nq * D, D, 1}, sk{n * Nk * D, Nk * D, D, 1};
    const jvp_strides_t ins[6] = {sq, sk, sk, sq, sk, sk}, outs[2] = {sq, sq};
    s = jvp_attn_fwd_dual(&cs, dtype, base + L.q, base + L.k, base + L.v, base + L.dq, base + L.dk,
                          base + L.dv, ins, mask, scale, base + L.o, base + L.t_o, outs,
                          lse ? reinterpret_cast<float*>(base + L.lse) : nullptr,
                          mu ? reinterpret_cast<float*>(base + L.mu) : nullptr, stream);
    if (s != JVP_OK) return s;
    last_path = t_last_path;
    if ((s = cu(cudaEventRecord(hp->computed[sl], stream), "cudaEventRecord")) != JVP_OK) return s;
    // device -> host
    if ((s = cu(cudaStreamWaitEvent(hp->out, hp->computed[sl], 0), "cudaStreamWaitEvent")) != JVP_OK)
      return s;
    struct { void* dst; size_t src, off, bytes; } back[4] = {
        {o, L.o, qoff, qbytes}, {t_o, L.t_o, qoff, qbytes},
        {lse, L.lse, static_cast<size_t>(lo * Nq) * sizeof(float), static_cast<size_t>(n * Nq) * sizeof(float)},
        {mu, L.mu, static_cast<size_t>(lo * Nq) * sizeof(float), static_cast<size_t>(n * Nq) * sizeof(float)}};
    for (auto& x : back) {
      if (!x.dst || x.bytes == 0) continue;
      s = cu(cudaMemcpyAsync(static_cast<uint8_t*>(x.dst) + x.off, base + x.src, x.bytes,
                             cudaMemcpyDeviceToHost, hp->out),
             "cudaMemcpyAsync (device to host)");
      if (s != JVP_OK) return s;
    }
    if ((s = cu(cudaEventRecord(hp->out_done[sl], hp->out), "cudaEventRecord")) != JVP_OK) return s;
  }
  // `stream` reaches this point only once every output is back on the host.
  if ((s = cu(cudaStreamWaitEvent(stream, hp->out_done[last_slot], 0), "cudaStreamWaitEvent")) != JVP_OK)
    return s;
  t_last_path = last_path;
  return ok();
}

// ---------------------------------------------------------------------------
// Backward without allocation (jvp_attn_bwd_dual_noalloc).
//
// Some callers cannot allocate device memory (plugins living in another
// framework's memory pool, code that must not call the allocator after
// start-up).  For them the backward's per-row scratch (nu and delta) lives in
// this fixed device array instead of a caller workspace.  Host code may not
// use the symbol itself as an address (it is a host-side stand-in); the real
// device address is looked up once per device and passed to the kernels.

static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[JVP_BWD_NOALLOC_SCRATCH_BYTES];

namespace jvp {
namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};  // device address of the array, per device

// Device address of the scratch array on the current device (first call per
// device: cudaGetSymbolAddress with that device current).
jvp_status_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(JVP_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(JVP_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
      return fail(JVP_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return JVP_OK;
}
}  // namespace
}  // namespace jvp

extern "C" jvp_status_t jvp_attn_bwd_dual_noalloc(
    const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q, const void* k, const void* v,
    const void* dq, const void* dk, const void* dv, const void* o, const void* t_o,
    const float* lse, const float* mu, const void* g_o, const void* g_to,
    const jvp_strides_t* in_strides, const jvp_mask_t* mask, float scale, void* g_q, void* g_k,
    void* g_v, void* g_dq, void* g_dk, void* g_dv, const jvp_strides_t* out_strides,
    void* stream) {
  if (!shape) return jvp::fail(JVP_ERR_INVALID_ARG, "shape is NULL");
  // (jvp_attn_bwd_dual_workspace_size returns SIZE_MAX for shapes whose
  // product of sizes overflows, so those are rejected here too)
  (void)dtype;
  if (shape->B > 0 && shape->H > 0 && shape->Nq > 0 &&
      jvp::bwd_base_workspace_size(shape) > JVP_BWD_NOALLOC_SCRATCH_BYTES)
    return jvp::fail(JVP_ERR_WORKSPACE,
                     "problem needs more than the 4 MiB fixed scratch of "
                     "jvp_attn_bwd_dual_noalloc (8 * B * H * Nq bytes); use jvp_attn_bwd_dual");
  void* scratch = nullptr;
  jvp_status_t s = jvp::noalloc_scratch(&scratch);
  if (s != JVP_OK) return s;
  const void* in[10] = {q, k, v, dq, dk, dv, o, t_o, g_o, g_to};
  void* out[6] = {g_q, g_k, g_v, g_dq, g_dk, g_dv};
  return bwd_dual_one_stream(shape, dtype, in, lse, mu, in_strides, mask, scale, out, out_strides,
                             scratch, JVP_BWD_NOALLOC_SCRATCH_BYTES, stream);
}

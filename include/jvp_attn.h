/*
 * jvp_attn.h -- C ABI of the GB300 attention forward + JVP library.
 *
 * The operation (the "JVP Flash Attention" project page, Description and Usage
 * sections): a drop-in for scaled_dot_product_attention(q, k, v, attn_mask)
 * whose dual forward `fwd_dual(q, k, v)`, used inside torch.func.jvp, returns
 * the attention output together with its forward-mode tangent.  Per (b, h):
 *
 *   S   = scale * Q K^T + M                 M: mask (see jvp_mask_t)
 *   P   = softmax over the kept keys of each row of S
 *   O   = P V
 *   dS  = scale * (dQ K^T + Q dK^T)         (M carries no tangent)
 *   mu  = rowsum(P * dS)                    (the tangent of the log-sum-exp)
 *   tO  = (P * dS) V - mu * O + P dV        (the directional derivative of O)
 *   lse = log sum_j exp(S_ij)               (natural log)
 *
 * A row that keeps no key yields O = tO = 0, lse = -inf and mu = 0.
 *
 * Conventions for every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *     allocates no device memory and keeps no pointer after the call returns.
 *   - Calls are asynchronous: work is enqueued on `stream` (a cudaStream_t
 *     passed as void*, NULL = the legacy default stream) and the call returns
 *     without synchronising.  Inputs must stay valid and unmodified, and outputs
 *     must not be read, until the stream reaches the work.
 *   - Tensors are [B, H, N, D] with element strides (jvp_strides_t); the
 *     innermost stride (d) must be 1.  Outputs must not overlap inputs.
 *   - Errors are reported by the returned status, never by abort or exception.
 *     Arguments are validated before anything is enqueued; on an error nothing
 *     is enqueued.  jvp_attn_last_error() gives a one-line reason (per thread).
 *   - A device-side wait that exceeds its time limit (about two seconds) makes
 *     the kernel return early and records JVP_ERR_DEVICE_TIMEOUT, which
 *     jvp_attn_get_device_status() reports.
 *   - Every size (B, H, Hkv, Nq, Nk, D) must be at most 2^31 - 1, and the
 *     products the launches form from them must fit too; larger problems are
 *     rejected with JVP_ERR_UNSUPPORTED before anything is enqueued.
 *   - The library caches, per device, device addresses of its own globals
 *     (the status word, the scratch of jvp_attn_bwd_dual_noalloc) the first
 *     time a device is used, and one non-blocking CUDA stream of its own (see
 *     jvp_attn_bwd_dual).  cudaDeviceReset() (or anything else that destroys
 *     the device's primary context) invalidates them: do not call the library
 *     on that device again in the same process after a reset.
 */
#ifndef JVP_ATTN_H_
#define JVP_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  JVP_OK = 0,
  JVP_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad stride, bad mask */
  JVP_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. D > 128, no sm_103 device) */
  JVP_ERR_ALIGNMENT = 3,      /* pointer or stride not aligned to the element size */
  JVP_ERR_CUDA = 4,           /* a CUDA runtime call failed (launch, attribute, ...) */
  JVP_ERR_DEVICE_TIMEOUT = 5, /* a device-side wait ran out (reported asynchronously) */
  JVP_ERR_WORKSPACE = 6,      /* workspace missing or too small */
  JVP_ERR_BOUNDS = 7          /* debug build only: a device-side bounds check failed
                                 (reported asynchronously, like a timeout) */
} jvp_status_t;

typedef enum { JVP_F32 = 0, JVP_F16 = 1, JVP_BF16 = 2 } jvp_dtype_t;

/* Mask kinds.  BOOL: uint8 elements, nonzero = the key takes part (SDPA's
 * boolean attn_mask).  ADDITIVE: float32 elements added to the scaled logits;
 * an entry of -inf excludes the key.  CAUSAL: key j takes part in row i iff
 * j <= i (top-left aligned); it uses no mask tensor (CAUSAL with a mask tensor
 * is rejected with JVP_ERR_INVALID_ARG).  BOOL_CAUSAL / ADDITIVE_CAUSAL: a
 * BOOL / ADDITIVE mask tensor and, in addition, the causal rule (SDPA rejects
 * is_causal together with attn_mask; these kinds are an extension, equal to
 * the mask tensor with the entries j > i excluded). */
typedef enum {
  JVP_MASK_NONE = 0,
  JVP_MASK_BOOL = 1,
  JVP_MASK_ADDITIVE = 2,
  JVP_MASK_CAUSAL = 3,
  JVP_MASK_BOOL_CAUSAL = 4,
  JVP_MASK_ADDITIVE_CAUSAL = 5
} jvp_mask_kind_t;

typedef struct {
  int64_t B, H; /* batch, query heads */
  int64_t Nq;   /* query rows */
  int64_t Nk;   /* key / value rows */
  int64_t D;    /* head dimension, 1..128 */
  int64_t Hkv;  /* key / value heads: 0 means H.  Otherwise H must be a multiple
                   of Hkv and query head h reads key / value head
                   h / (H / Hkv) (grouped-query attention). */
} jvp_shape_t;

/* Element strides of a [B, H, N, D] tensor; d must be 1. */
typedef struct {
  int64_t b, h, n, d;
} jvp_strides_t;

/* Mask of logical shape [B|1, H|1, Nq, Nk]; stride 0 broadcasts a dimension
 * (e.g. stride_h = 0 for a mask shared by all heads).  `ptr` is NULL for
 * JVP_MASK_NONE and JVP_MASK_CAUSAL. */
typedef struct {
  int32_t kind; /* jvp_mask_kind_t */
  const void* ptr;
  int64_t stride_b, stride_h, stride_q, stride_k;
} jvp_mask_t;

/*
 * Fused attention forward + JVP (the project page's `JVPAttn.fwd_dual`).
 *
 *   shape          sizes; B*H*Nq == 0 or Nk == 0 is valid (nothing to compute
 *                  beyond writing the empty-row convention when Nk == 0).
 *   dtype          element type shared by q, k, v, dq, dk, dv, o and t_o.
 *   q, dq          [B,H,Nq,D];  k, v, dk, dv [B,Hkv,Nk,D]  (device, read only).
 *   in_strides     6 stride records, in the order q, k, v, dq, dk, dv.
 *   mask           NULL or a mask description (see jvp_mask_t).
 *   scale          logit scale (SDPA's default is 1/sqrt(D)); must be finite.
 *   o, t_o         [B,H,Nq,D] outputs (device, written).
 *   out_strides    2 stride records, for o and t_o.
 *   lse, mu        NULL or [B,H,Nq] contiguous float32 outputs (device).
 *   stream         cudaStream_t as void*.
 *
 * fp16/bf16 inputs with D a multiple of 8 up to 128, 16-byte aligned base
 * pointers and strides take the tensor-core path (TMA + tcgen05 + TMEM, fp32
 * accumulation; D <= 64 runs the D = 64 kernel and larger D the D = 128
 * kernel, on zero-filled columns past D); every other valid case (float32,
 * other D) takes the CUDA-core path, which computes in fp32 FFMA.
 */
jvp_status_t jvp_attn_fwd_dual(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                               const void* k, const void* v, const void* dq, const void* dk,
                               const void* dv, const jvp_strides_t* in_strides,
                               const jvp_mask_t* mask, float scale, void* o, void* t_o,
                               const jvp_strides_t* out_strides, float* lse, float* mu,
                               void* stream);

/*
 * jvp_attn_fwd_dual with a caller-provided workspace, which lets the
 * tensor-core path split the key range of small problems (fewer query tiles
 * than SMs) over several CTAs and merge their partial softmax states in a
 * second kernel (split-KV; the associative merge of (max, sums, A, T) states).
 * Results equal jvp_attn_fwd_dual's up to floating-point rounding order.
 *
 *   workspace        NULL, or device scratch of workspace_bytes bytes, 16-byte
 *                    aligned, owned by the caller; contents on entry do not
 *                    matter.  The split runs only if workspace_bytes is at
 *                    least jvp_attn_fwd_dual_workspace_size(shape, dtype);
 *                    otherwise (or with NULL) the call is jvp_attn_fwd_dual.
 *   other arguments  as for jvp_attn_fwd_dual.
 *
 * Calls that share a workspace and overlap on the GPU race on it.
 */
jvp_status_t jvp_attn_fwd_dual_ws(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                                  const void* k, const void* v, const void* dq, const void* dk,
                                  const void* dv, const jvp_strides_t* in_strides,
                                  const jvp_mask_t* mask, float scale, void* o, void* t_o,
                                  const jvp_strides_t* out_strides, float* lse, float* mu,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes with which jvp_attn_fwd_dual_ws splits the key range of
 * `shape` on the current device: splits * B*H*Nq * (16 + 8 D) bytes, or 0 when
 * the problem is not split (enough query tiles to fill the SMs, too few keys,
 * a shape the tensor-core path does not take, or no device). */
size_t jvp_attn_fwd_dual_workspace_size(const jvp_shape_t* shape, jvp_dtype_t dtype);

/*
 * jvp_attn_fwd_dual for inputs and outputs in HOST memory (the end-to-end
 * form of the call: copies included).  The B*H (batch, head) pairs are split
 * into `chunks` groups; each group's inputs are copied into one of two device
 * staging slots (in `workspace`) on a copy stream of the library, the fused
 * kernel runs on `stream`, and the outputs go back on a second copy stream,
 * so one group's copies overlap the neighbouring groups' kernels.
 *
 *   q, k, v, dq, dk, dv   HOST pointers to contiguous [B,H,Nq|Nk,D] tensors;
 *                         page-locked (pinned) memory lets the copies run
 *                         asynchronously and overlap.
 *   o, t_o                HOST pointers to contiguous [B,H,Nq,D] outputs.
 *   lse, mu               NULL or HOST pointers to [B,H,Nq] float32 outputs.
 *   mask                  as for jvp_attn_fwd_dual, but a mask tensor must be
 *                         a DEVICE tensor shared by every (batch, head)
 *                         (stride_b = stride_h = 0).
 *   chunks                number of groups (>= 1, at most B*H are used; more
 *                         groups overlap more but launch smaller kernels).
 *                         Group sizes fall linearly (one pair each plus shares
 *                         weighted G, G-1, ..., 1 of the rest), so the last
 *                         group -- whose kernel and copies back are all that
 *                         follows the last copy in -- is the smallest.
 *   workspace             DEVICE scratch of at least
 *                         jvp_attn_fwd_dual_host_workspace_size(shape, dtype,
 *                         chunks) bytes, 256-byte aligned, owned by the caller.
 *   stream                the call is ordered after the work already on
 *                         `stream`, and `stream` reaches its end only when
 *                         every output is in host memory: synchronise
 *                         `stream` before reading them.  Inputs must stay
 *                         unchanged until then.
 *
 * Grouped-query attention (Hkv != H) is not taken here.  Calls from several
 * host threads are serialised while they enqueue; calls that share a
 * workspace must be ordered (e.g. on one stream).
 */
jvp_status_t jvp_attn_fwd_dual_host(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                                    const void* k, const void* v, const void* dq, const void* dk,
                                    const void* dv, const jvp_mask_t* mask, float scale, void* o,
                                    void* t_o, float* lse, float* mu, int chunks,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Device staging bytes jvp_attn_fwd_dual_host needs: two slots, each holding
 * the largest group's six inputs, two outputs, lse and mu (0 for an invalid
 * shape). */
size_t jvp_attn_fwd_dual_host_workspace_size(const jvp_shape_t* shape, jvp_dtype_t dtype,
                                             int chunks);

/*
 * Attention forward without tangents (the project page's `jvp_attention` /
 * `attention`, Usage section): O = softmax(scale Q K^T + M) V and lse.
 * Arguments as for jvp_attn_fwd_dual; in_strides holds 3 records (q, k, v)
 * and out_strides 1 record (o).
 */
jvp_status_t jvp_attn_fwd(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                          const void* k, const void* v, const jvp_strides_t* in_strides,
                          const jvp_mask_t* mask, float scale, void* o,
                          const jvp_strides_t* out_strides, float* lse, void* stream);

/*
 * Reverse mode of the dual computation (the backward needed to train through
 * `fwd_dual` or to form Hessian-vector products: the project page,
 * Description and Results sections).  Given the cotangents g_o, g_to of
 * Loss = <g_o, O> + <g_to, tO>, writes the gradients with respect to q, k, v,
 * dq, dk, dv.  No gradient flows into the mask.
 *
 *   q, k, v, dq, dk, dv   the forward inputs (as passed to jvp_attn_fwd_dual)
 *   o, t_o, lse, mu       that call's outputs (lse and mu are required here)
 *   g_o, g_to             cotangents, [B,H,Nq,D]
 *   in_strides            10 records: q, k, v, dq, dk, dv, o, t_o, g_o, g_to
 *   g_q, g_k, g_v, g_dq, g_dk, g_dv   outputs, shapes of q, k, v, dq, dk, dv
 *                         (with grouped-query attention g_k, g_v, g_dk, g_dv
 *                         sum the contributions of every query head of the
 *                         group)
 *   out_strides           6 records in that order
 *   workspace             device scratch of at least 8 * B * H * Nq bytes
 *                         (nu and delta per query row), 4-byte aligned, owned
 *                         by the caller; its contents on entry do not matter
 *                         and are overwritten.  With the (larger, 16-byte
 *                         aligned) jvp_attn_bwd_dual_workspace_size() bytes,
 *                         problems whose key-major CTAs would fill less than
 *                         half of the SMs and each walk 64+ query tiles (few
 *                         key/value heads) share each key tile's query tiles
 *                         among several CTAs, and likewise each query tile's
 *                         key tiles when few query-major CTAs walk 64+ key
 *                         tiles (few queries, many keys); a combine kernel
 *                         adds the fp32 partial sums on the same stream
 *                         (results differ from the unsplit kernels only by
 *                         the order of fp32 additions).
 *
 * Every tensor has the same dtype; mask and scale as in the forward call.
 * fp16/bf16 with D a multiple of 8 up to 128 and 16-byte aligned tensors run
 * a row pass and tcgen05 kernels (query-major for g_q, g_dq; key-major for
 * g_k, g_dk, g_v, g_dv), fp32 accumulation (the D = 64 or 128 kernels, with
 * zero-filled columns past D); every other case runs three CUDA-core kernels
 * in fp32.  All work is ordered on `stream`: the key-major kernels run on a
 * stream the library owns (one per device, created on first use), which waits
 * for the row pass through an event, and `stream` waits for them through
 * another event before anything enqueued after this call, so the two
 * kernels overlap and the caller sees one stream (this fork and join also
 * records into a stream capture; make the first backward call on a device
 * outside any capture, since it creates that stream).  Returns
 * JVP_ERR_WORKSPACE if the workspace is NULL or too small.
 */
jvp_status_t jvp_attn_bwd_dual(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                               const void* k, const void* v, const void* dq, const void* dk,
                               const void* dv, const void* o, const void* t_o, const float* lse,
                               const float* mu, const void* g_o, const void* g_to,
                               const jvp_strides_t* in_strides, const jvp_mask_t* mask,
                               float scale, void* g_q, void* g_k, void* g_v, void* g_dq,
                               void* g_dk, void* g_dv, const jvp_strides_t* out_strides,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes jvp_attn_bwd_dual takes for `shape` on the current device:
 * 8 * B * H * Nq, rounded up to 256, plus ks * 4 * B * Hkv * Nk * D' * 4
 * bytes when the tensor-core kernels split the key side of this shape into ks
 * parts and qs * 2 * B * H * Nq * D' * 4 bytes when they split the query side
 * into qs (D' = 64 for D <= 64, else 128; ks and qs from the SM count).  0 for a NULL
 * shape or a negative size, SIZE_MAX for a shape too large for any launch (a
 * size above 2^31 - 1, or B * H * Nq above it). */
size_t jvp_attn_bwd_dual_workspace_size(const jvp_shape_t* shape, jvp_dtype_t dtype);

/*
 * Reverse mode of attention without tangents: the backward that
 * `jvp_attention` needs when it is used as a plain drop-in for
 * scaled_dot_product_attention (the project page, Usage section) and trained
 * by ordinary back-propagation.  Given the cotangent g_o of Loss = <g_o, O>,
 * writes the gradients with respect to q, k, v; no gradient flows into the
 * mask.  It is the dual backward with dq = dk = dv = 0 and g_to = 0, without
 * the work those zeros would cost:
 *   P = exp(S - lse), delta = rowsum(g_o * O), gP = g_o V^T,
 *   gS = P * (gP - delta), g_q = scale gS K, g_k = scale gS^T Q, g_v = P^T g_o.
 *
 *   q, k, v        the forward inputs (as passed to jvp_attn_fwd)
 *   o, lse         that call's outputs (lse is required)
 *   g_o            cotangent, [B,H,Nq,D]
 *   in_strides     5 records: q, k, v, o, g_o
 *   g_q, g_k, g_v  outputs, shapes of q, k, v (with grouped-query attention
 *                  g_k, g_v sum the contributions of every query head of the
 *                  group); out_strides 3 records in that order
 *   workspace      device scratch of at least jvp_attn_bwd_workspace_size()
 *                  bytes, 4-byte aligned, owned by the caller; its contents on
 *                  entry do not matter and are overwritten.
 *
 * Every tensor has the same dtype; mask and scale as in the forward call.
 * fp16/bf16 with D a multiple of 8 up to 128 and 16-byte aligned tensors run
 * a row pass and two tcgen05 kernels (query-major for g_q; key-major for g_k and
 * g_v in one pass at every D, on the library's second stream as in
 * jvp_attn_bwd_dual); every other case runs three CUDA-core kernels in fp32.
 * All work is ordered on `stream`.  Returns JVP_ERR_WORKSPACE if the
 * workspace is NULL or too small.
 */
jvp_status_t jvp_attn_bwd(const jvp_shape_t* shape, jvp_dtype_t dtype, const void* q,
                          const void* k, const void* v, const void* o, const float* lse,
                          const void* g_o, const jvp_strides_t* in_strides,
                          const jvp_mask_t* mask, float scale, void* g_q, void* g_k, void* g_v,
                          const jvp_strides_t* out_strides, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Workspace bytes jvp_attn_bwd takes for `shape` (the same as
 * jvp_attn_bwd_dual_workspace_size; 8 * B * H * Nq bytes suffice, without the
 * key-major split). */
size_t jvp_attn_bwd_workspace_size(const jvp_shape_t* shape, jvp_dtype_t dtype);

/*
 * jvp_attn_bwd_dual for callers that cannot allocate device memory.  The
 * pages have no counterpart to this entry point; it exists for callers such
 * as plugins that run inside someone else's process or memory pool, code
 * paths that must not touch the allocator after start-up, and callers without
 * access to cudaMalloc.  It allocates nothing: instead of a caller-provided
 * workspace it uses a fixed scratch array that the library itself places in
 * device memory (4 MiB, JVP_BWD_NOALLOC_SCRATCH_BYTES; every device that loads
 * the library holds it until the process exits).  Arguments are those of
 * jvp_attn_bwd_dual without the workspace.
 *
 *   - Size limit: the problem may need at most 4 MiB of scratch, i.e.
 *     8 * B * H * Nq <= 4 MiB (B * H * Nq <= 524288 query rows in total).
 *     Larger problems return JVP_ERR_WORKSPACE with a message naming the limit.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (with that device current) and caches it; make that first call
 *     before any stream capture.
 *   - Streams: every kernel runs on `stream` (no second stream, no events).
 *   - Sharing: every call uses the same array.  Nothing in it needs to start
 *     at zero (each call overwrites the part it reads), but calls whose work
 *     overlaps on the GPU (different streams, no ordering between them) race
 *     on it; order them, e.g. issue them on one stream.
 */
#define JVP_BWD_NOALLOC_SCRATCH_BYTES (4u << 20)
jvp_status_t jvp_attn_bwd_dual_noalloc(const jvp_shape_t* shape, jvp_dtype_t dtype,
                                       const void* q, const void* k, const void* v,
                                       const void* dq, const void* dk, const void* dv,
                                       const void* o, const void* t_o, const float* lse,
                                       const float* mu, const void* g_o, const void* g_to,
                                       const jvp_strides_t* in_strides, const jvp_mask_t* mask,
                                       float scale, void* g_q, void* g_k, void* g_v, void* g_dq,
                                       void* g_dk, void* g_dv, const jvp_strides_t* out_strides,
                                       void* stream);

/*
 * Synchronises `stream`, then returns and clears the device-side status word:
 * JVP_ERR_BOUNDS if a kernel of a debug build of the library found an index
 * out of its bounds (and skipped that access), else JVP_ERR_DEVICE_TIMEOUT if
 * any kernel gave up on a wait since the last call, JVP_ERR_CUDA if the
 * stream reports an error, else JVP_OK.
 */
jvp_status_t jvp_attn_get_device_status(void* stream);

/* Static string for a status code. */
const char* jvp_attn_status_string(jvp_status_t status);

/* One-line description of the last error returned on the calling thread. */
const char* jvp_attn_last_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int jvp_attn_version(void);

/*
 * Diagnostic: enqueues a one-thread kernel that waits on a device barrier
 * that nothing completes, with a wait limit of `limit_cycles` SM clock cycles,
 * so that the bounded-wait path runs out and records JVP_ERR_DEVICE_TIMEOUT
 * without faulting or hanging the GPU.  limit_cycles must be in [1, 2^31).
 */
jvp_status_t jvp_attn_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/*
 * Diagnostic: which kernel family the last successful call on the calling
 * thread enqueued: 1 = tensor-core path, 2 = CUDA-core path, 3 = tensor-core
 * path with split-KV and the merge kernel, 4 = tensor-core path with each
 * query tile's key range split between the two CTAs of a cluster (small
 * problems at D <= 64; no workspace), 0 = nothing was enqueued (empty
 * problem or an error).
 */
int jvp_attn_debug_last_path(void);

/*
 * Diagnostic: enable = 1 (the default) lets jvp_attn_fwd_dual split the key
 * range of small problems between the two CTAs of a cluster (path 4 above);
 * enable = 0 keeps later calls (process-wide) on the single pass.  Both give
 * the same function up to floating-point rounding order; this exists so that
 * tests and benchmarks can compare them.  Returns JVP_ERR_INVALID_ARG for
 * other values.
 */
jvp_status_t jvp_attn_debug_set_cluster_split(int enable);

#ifdef __cplusplus
}
#endif

#endif /* JVP_ATTN_H_ */

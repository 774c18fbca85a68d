/*
 * jllm_q4k.h -- C ABI of the GB300 (sm_103a) Q4_K dequant-fused matmul library.
 *
 * The library computes Y[M,N] = X[M,K] * dequant(W)[N,K]^T where W is a weight
 * matrix stored as GGUF Q4_K super-blocks and X is fp16.  This is the work of
 * the two kernels the genie-ai-runtime README lists under "At a glance"
 * (Kernels bullet) and "Project layout" (src/kernels/): the "INT4
 * dequant-fused GEMV" used for decode (M = 1) and the "tensor-core MMQ Q4_K
 * prefill" used for prompts (M = prompt tokens); and of the SwiGLU and RMSNorm
 * parts of its "fused RMSNorm + RoPE + SwiGLU" kernel.  The pages say the runtime loads
 * GGUF Q4_K_M models ("At a glance", Models bullet) but print neither the
 * block layout nor any kernel interface; both are defined here.
 *
 * ---------------------------------------------------------------- layouts --
 * Q4_K super-block (144 bytes, 256 weights), public GGUF layout:
 *   bytes 0..1    d     fp16 little endian        (scale of the 6-bit scales)
 *   bytes 2..3    dmin  fp16 little endian        (scale of the 6-bit mins)
 *   bytes 4..15   s[12] eight 6-bit scales sc_j and eight 6-bit mins m_j:
 *                   j<4 : sc_j = s[j] & 63,  m_j = s[j+4] & 63
 *                   j>=4: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4
 *                         m_j  = (s[j+4] >> 4) | (s[j]   >> 6) << 4
 *   bytes 16..143 qs[128] 4-bit codes q: weight 64c+l (c = 0..3, l = 0..31) is
 *                 the low nibble of qs[32c+l], weight 64c+32+l its high nibble.
 *   value of weight i (sub-block j = i/32): w = d*sc_j*q - dmin*m_j.
 * W   : [N rows][K/256 blocks] of 144-byte blocks, rows contiguous (row pitch
 *       K/256*144 bytes), device memory, 16-byte aligned.
 * X   : [M][K] fp16 row-major, contiguous, device memory, 16-byte aligned.
 * Y   : [M][N] row-major, contiguous, fp32 or fp16, device memory,
 *       16-byte aligned.
 * K must be a positive multiple of 256; M, N >= 1.  Sizes are element counts.
 *
 * ---------------------------------------------------------------- numerics --
 * Dequant: fp32 output is d*sc*q - dmin*m evaluated in fp32 in that order
 * (the three products are exact, the difference rounds once); fp16 output is
 * that fp32 value rounded to nearest even.  Matmul outputs satisfy, per
 * element, |y - y_ref| <= 2e-3 * sum_k |x_k * w_nk| + 1e-5 against the exact
 * product of the fp16 X and the exact dequantised W.
 *
 * --------------------------------------------------------------- semantics --
 * Every pointer argument is caller-owned device memory unless stated; the
 * library never allocates or frees device memory on these calls.  `stream` is
 * a cudaStream_t (NULL = legacy default stream).  Argument errors are
 * reported synchronously, before anything is launched; otherwise the work is
 * enqueued on `stream` and the call returns JLLM_OK without synchronising.
 * A launch failure returns JLLM_ERR_CUDA.  Kernel-side waits are bounded: a
 * wait that runs out sets a device error word that jllm_get_device_error()
 * reads.  No call throws or prints.  State kept: cached device properties,
 * the CUDA driver's tensor-map encoder, a table of the 64 most recently used
 * encoded tensor maps (keyed by device, address, extents and tile; guarded by
 * a mutex), and the static workspace of jllm_q4k_gemm_noalloc.  Environment variables read (once per process):
 * JLLM_PDL, JLLM_GEMV_MAX_M and JLLM_GEMM_MMA_MAX_M, described below; no
 * other setting changes launch shapes or summation order.
 * The GEMV and GEMM kernels are launched with programmatic dependent launch:
 * they start fetching W while the kernel enqueued just before them on the
 * same stream is still running, and read X / write Y (and the workspace)
 * only after it has completed.  So W must not be written by that immediately
 * preceding kernel (weights written earlier in the stream are fine).  Setting
 * the environment variable JLLM_PDL=0 (read once per process) launches them
 * without it.
 */
#ifndef JLLM_Q4K_H
#define JLLM_Q4K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  JLLM_OK = 0,
  JLLM_ERR_INVALID_ARG = 1,       /* NULL pointer, M/N < 1, bad enum value      */
  JLLM_ERR_UNSUPPORTED_SHAPE = 2, /* K not a positive multiple of 256, or a
                                     size beyond the kernels' index range      */
  JLLM_ERR_MISALIGNED = 3,        /* a pointer not 16-byte aligned             */
  JLLM_ERR_UNSUPPORTED_DTYPE = 4, /* output dtype not allowed for this call    */
  JLLM_ERR_WORKSPACE = 5,         /* workspace too small or misaligned */
  JLLM_ERR_CUDA = 6,              /* a CUDA runtime/driver call failed         */
  JLLM_ERR_DEVICE_TIMEOUT = 7,    /* a kernel-side bounded wait ran out        */
  JLLM_ERR_NO_DEVICE = 8          /* the current device is not sm_103          */
} jllm_status;

typedef enum { JLLM_F32 = 0, JLLM_F16 = 1 } jllm_dtype;

/* A cudaStream_t, passed as an opaque pointer. */
typedef void* jllm_stream_t;

/*
 * jllm_q4k_dequant -- expand W to an [N,K] row-major matrix.
 *   w_q4k  : W, [N][K/256] blocks (see layouts)
 *   out    : [N][K] fp32 or fp16 (out_dt), 16-byte aligned
 * Result is bit-exact to the rule under "numerics".
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, UNSUPPORTED_DTYPE, CUDA.
 */
jllm_status jllm_q4k_dequant(const void* w_q4k, void* out, jllm_dtype out_dt, int64_t N,
                             int64_t K, jllm_stream_t stream);

/*
 * jllm_q4k_gemv -- decode matmul, M = 1: y[n] = sum_k x[k] * w[n,k].
 * (the README's "INT4 dequant-fused GEMV", Kernels bullet)
 *   w_q4k : W, [N][K/256] blocks
 *   x     : [K] fp16
 *   y     : [N] fp32
 *   ws, ws_bytes : unused by the GEMV (jllm_q4k_workspace_bytes(1, N, K)
 *           is 0); may be NULL/0
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, WORKSPACE, CUDA.
 */
jllm_status jllm_q4k_gemv(const void* w_q4k, const void* x, float* y, int64_t N, int64_t K,
                          void* ws, size_t ws_bytes, jllm_stream_t stream);

/*
 * jllm_q4k_gemv_batch -- count (1..8) decode GEMVs that read the same x, in
 * one launch: y[i][n] = sum_k x[k] * w_i[n,k] for n < N[i].  The pages name
 * no such call; it serves the matrices of a decoder layer that share an
 * input (q, k, v; gate, up), so that they cost one dependent launch.
 *   w_q4k : host array of count device pointers, W_i [N[i]][K/256] blocks
 *   y     : host array of count device pointers, [N[i]] fp32 each
 *   N     : host array of count row counts
 *   x     : [K] fp16, shared
 * The host arrays are read before the call returns.  Each y[i] equals
 * jllm_q4k_gemv(w_q4k[i], x, y[i], N[i], K) within the matmul bound (the
 * launch configuration follows the total row count, so the fp32 summation
 * order may differ from a single call's).
 * Errors: INVALID_ARG (also count outside 1..8), UNSUPPORTED_SHAPE,
 *         MISALIGNED, CUDA.
 */
jllm_status jllm_q4k_gemv_batch(const void* const* w_q4k, float* const* y, const int64_t* N, int count,
                                const void* x, int64_t K, jllm_stream_t stream);

/*
 * jllm_q4k_gemv_rmsnorm_batch -- jllm_q4k_gemv_batch on the RMS-normalised x:
 *   xn[k] = fp16( x[k] * r * gamma[k] ),  r = 1 / sqrt(sum_k x[k]^2 / K + eps)
 *   y[i][n] = sum_k xn[k] * w_i[n,k]
 * The RMSNorm of the README's "fused RMSNorm + RoPE + SwiGLU" kernel (At a
 * glance, Kernels bullet), fused into the prologue of the decode GEMV so that
 * a decoder layer's q/k/v (and gate/up) launch reads the residual stream
 * directly.  The pages print no formula; this is the standard RMSNorm.
 *   x     : [K] fp16, shared; gamma: [K] fp32 (16-byte aligned); eps in [0, 1]
 *   w_q4k, y, N, count: as jllm_q4k_gemv_batch
 * gamma, like the weights, is read before the wait on the previous kernel in
 * the stream (see the PDL paragraph above): it must not be written by that
 * kernel.
 * Every CTA forms r itself (fp32 sum of exact fp16 squares in a fixed order,
 * then 1/sqrt), so r is the same for all outputs.  The normalised x is
 * rounded to fp16 (the GEMV's input type) before the products; y is within
 * the matmul bound of the exact xn with one extra 2^-11 relative term for
 * that rounding, which the bound covers.
 * Errors: INVALID_ARG (also count outside 1..8, eps outside [0, 1] or NaN),
 *         UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
jllm_status jllm_q4k_gemv_rmsnorm_batch(const void* const* w_q4k, float* const* y, const int64_t* N,
                                        int count, const void* x, const float* gamma, float eps,
                                        int64_t K, jllm_stream_t stream);

/*
 * jllm_q4k_gemv_qkv_rope -- the q, k and v projections of one decode token in
 * one launch, with the rotary position embedding applied to q and k in the
 * epilogue: the RoPE of the README's "fused RMSNorm + RoPE + SwiGLU" kernel
 * (At a glance, Kernels bullet).  The pages print no rotary formula; this is
 * the form of the Qwen3 model they run:
 *   xn     = x, or the RMSNorm of x when gamma != NULL (as in
 *            jllm_q4k_gemv_rmsnorm_batch)
 *   q, k   = dequant(Wq) xn, dequant(Wk) xn; v = dequant(Wv) xn
 *   per head h of q (and of k), 128 values t[0..127]:
 *     optional per-head RMSNorm: t = t * g / sqrt(sum(t^2)/128 + head_eps),
 *       g = q_gamma (resp. k_gamma) [128], skipped when that pointer is NULL
 *     rotation of pairs (j, j+64), j < 64, by a = pos * rope_base^(-2j/128):
 *       out[j] = t[j] cos a - t[j+64] sin a;  out[j+64] = t[j+64] cos a + t[j] sin a
 *   w_q4k : host array of 3 device pointers: Wq [n_q_heads*128][K/256]
 *           blocks, Wk and Wv [n_kv_heads*128][K/256] blocks
 *   y     : host array of 3 device pointers: q [n_q_heads*128], k and v
 *           [n_kv_heads*128], fp32 (q, k rotated; v plain)
 *   x     : [K] fp16; gamma: [K] fp32 or NULL, eps in [0, 1]
 *   q_gamma, k_gamma: [128] fp32 or NULL; head_eps in [0, 1]
 *   pos   : token position (any 32-bit value); rope_base > 0 (Qwen3: 1e6)
 * Head size 128 only.  base^(-2j/128) is formed on the host in fp64, the angle
 * and its reduction modulo 2 pi in fp64, the cosine and sine in fp32; each q/k
 * value stays within the matmul bound propagated through the norm and the
 * rotation.  The 8 CTAs that compute one head form
 * a thread-block cluster and reduce the head's sum of squares through
 * distributed shared memory.  gamma, q_gamma and k_gamma, like the weights,
 * must not be written by the kernel enqueued just before (PDL paragraph).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
jllm_status jllm_q4k_gemv_qkv_rope(const void* const* w_q4k, float* const* y, int64_t n_q_heads,
                                   int64_t n_kv_heads, const void* x, int64_t K, const float* gamma,
                                   float eps, const float* q_gamma, const float* k_gamma, float head_eps,
                                   int64_t pos, float rope_base, jllm_stream_t stream);

/*
 * jllm_q4k_gemv_chain -- a sequence of decode GEMV steps in ONE persistent
 * launch (one CTA per SM, all resident: a cooperative launch).  Step s is
 * count (1..4) GEMVs over one x: y_i[n] = sum_k x[k] * w_i[n,k], n < N[i].
 * The steps run in order: step s+1 reads its x only after every y of steps
 * 0..s is written, so a step may read an earlier step's y (with y_f16 = 1
 * it is directly an fp16 x).  Weights are streamed ahead of the steps,
 * across step boundaries.  The pages name no such call: it is the decode
 * sweep of the README's "INT4 dequant-fused GEMV" (At a glance, Kernels
 * bullet) -- a layer's q/k/v, o, gate/up and down projections, layer after
 * layer -- without a launch per matmul.
 *   steps  : host array of n_steps (1..JLLM_CHAIN_MAX_STEPS) descriptors,
 *            read before the call returns (the launch keeps a copy)
 *     count  : 1..JLLM_CHAIN_MAX_MATS
 *     y_f16  : 0 = y fp32, 1 = y fp16 (round to nearest even)
 *     K      : a multiple of 256, at most JLLM_CHAIN_MAX_K
 *     x      : [K] fp16, device, 16-byte aligned
 *     w_q4k[i], y[i], N[i] : W_i [N[i]][K/256] blocks, its output [N[i]],
 *            both device and 16-byte aligned; N[i] >= 0 (0: the entry is
 *            skipped and its pointers are not read)
 *   sync   : device, jllm_q4k_gemv_chain_sync_bytes(n_steps) bytes, 4-byte
 *            aligned, zero before the first call (cudaMemset); a call that
 *            completes leaves it zero.  One sync buffer serves one call at a
 *            time (not two chains that may run concurrently).
 * The launch holds one CTA on every SM (about 221 KiB of shared memory each)
 * for its whole duration; CTAs wait on one another's step counters, so other
 * work on the device can delay it (a wait that runs out after 2 s is reported
 * by jllm_get_device_error) but not change its results.
 * Each y equals jllm_q4k_gemv's within the matmul bound (the split of K and
 * the summation order differ).  No W of any step may be written by an
 * earlier step of the same call nor by the kernel enqueued just before it.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA (also when the
 *         device cannot hold one CTA per SM).  A bounded wait that runs out
 *         is reported by jllm_get_device_error; sync must then be zeroed
 *         again before the next call.
 */
#define JLLM_CHAIN_MAX_STEPS 256
#define JLLM_CHAIN_MAX_MATS 4
#define JLLM_CHAIN_MAX_K 12288
typedef struct {
  int32_t count;
  int32_t y_f16;
  int64_t K;
  const void* x;
  const void* w_q4k[JLLM_CHAIN_MAX_MATS];
  void* y[JLLM_CHAIN_MAX_MATS];
  int64_t N[JLLM_CHAIN_MAX_MATS];
} jllm_gemv_step;
jllm_status jllm_q4k_gemv_chain(const jllm_gemv_step* steps, int n_steps, uint32_t* sync, jllm_stream_t stream);

/* Bytes of the sync buffer of a chain of n_steps steps (0 outside 1..JLLM_CHAIN_MAX_STEPS). */
size_t jllm_q4k_gemv_chain_sync_bytes(int n_steps);

/*
 * jllm_q4k_gemm -- Y[M,N] = X[M,K] * dequant(W)^T for any M >= 1.
 * (the README's "tensor-core MMQ Q4_K prefill" for M above the GEMV
 *  threshold, the GEMV kernel at or below it)
 *   w_q4k : W, [N][K/256] blocks
 *   x     : [M][K] fp16
 *   y     : [M][N], fp32 or fp16 (y_dt)
 *   ws, ws_bytes : optional workspace (see jllm_q4k_workspace_bytes)
 * M <= jllm_q4k_gemv_max_m() runs the GEMV kernel (gemm(M=1) == gemv).
 * A few tokens (M <= 24, or M <= 40 when W has at most 64 tiles of 128 rows,
 * counted over all matrices of a batch) run the few-token kernel: warp-level
 * tensor cores (mma.sync, fp16 operands, fp32 accumulation) on weights
 * dequantised in registers in the factored form d*sc*q - dmin*m (the code
 * products exact, the min term as exact fp16 hi + lo parts against hi + lo
 * sub-block sums of x), K split over a thread-block cluster whose partials
 * are added in a fixed order through distributed shared memory (no
 * workspace; deterministic).  Its domain: |dmin*m| <= 65504 and every sum of
 * x over 32 consecutive values of a super-block <= 65504 in magnitude.  The
 * environment variable JLLM_GEMM_MMA_MAX_M (0..40, read once per process)
 * replaces that rule: M up to its value take the few-token kernel whatever
 * the shape, larger M the tcgen05 kernel.
 * Larger M runs the TMA + tcgen05 kernel (fp16 dequantised W, fp32
 * accumulation in tensor memory).  With a workspace the tcgen05 kernel
 * shares the K steps of the last wave of tiles evenly among the SMs
 * (stream-K); the cut tiles' fp32 partials are added in a fixed order, so
 * results are deterministic for a given device.  Tiles of at most 128
 * tokens that number fewer than the SMs are instead split along K over a
 * thread-block cluster of up to 8 CTAs (partials added in K order through
 * distributed shared memory, no workspace); the split depends on the
 * launch's tile count, so a batched call and single calls may differ in
 * the last bits.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, UNSUPPORTED_DTYPE,
 *         WORKSPACE, CUDA.
 */
jllm_status jllm_q4k_gemm(const void* w_q4k, const void* x, void* y, jllm_dtype y_dt, int64_t M,
                          int64_t N, int64_t K, void* ws, size_t ws_bytes, jllm_stream_t stream);

/*
 * jllm_q4k_gemm_noalloc -- jllm_q4k_gemm with the library's own workspace.
 * The pages describe no such call; it exists for callers that cannot hand
 * the library device memory.  The workspace is a static device array in
 * the library image (zero at load, ~42 MB, enough for up to 160 SMs),
 * found with cudaGetSymbolAddress once per device; nothing is allocated.
 * Arguments and results as jllm_q4k_gemm without ws/ws_bytes.  The array
 * is shared by every call on a device, so calls must not overlap: issue
 * them on one stream (or order them), as with one caller workspace.
 * The array belongs to the tcgen05 GEMM's module, so it is resident on
 * every device that runs any tcgen05 GEMM of this library, whether or not
 * this entry point is called.  Recovery: every call that completes leaves
 * the array reusable; after a kernel-side timeout, jllm_get_device_error()
 * (which reports it) also returns the array's flag words to zero, so call
 * it before the next call on that device.
 * Errors: as jllm_q4k_gemm; WORKSPACE if the device has more SMs than the
 * array was sized for.
 */
jllm_status jllm_q4k_gemm_noalloc(const void* w_q4k, const void* x, void* y, jllm_dtype y_dt,
                                  int64_t M, int64_t N, int64_t K, jllm_stream_t stream);

/*
 * jllm_q4k_gemm_batch -- count (1..4) prefill GEMMs that read the same X,
 * in one launch: Y_i[M,N[i]] = X[M,K] * dequant(W_i)^T.  The pages name no
 * such call; it serves the matrices of a decoder layer that share an input
 * (q, k, v; gate, up), so that the small ones (k, v) share the SMs with
 * the large one instead of each paying a launch and a tail.
 *   w_q4k : host array of count device pointers, W_i [N[i]][K/256] blocks
 *   x     : [M][K] fp16, shared
 *   y     : host array of count device pointers, [M][N[i]] each, fp32 or
 *           fp16 (y_dt, one type for all)
 *   N     : host array of count row counts
 *   ws, ws_bytes : optional workspace, sized by
 *           jllm_q4k_workspace_bytes(M, sum N[i], K)
 * The host arrays are read before the call returns.  M above the GEMV
 * threshold runs one launch over the tiles of all matrices, matrix by
 * matrix: the few-token kernel where jllm_q4k_gemm's rule picks it for the
 * batch's total rows, else one persistent tcgen05 launch (with a workspace
 * the stream-K split covers them all); at or below the threshold, one GEMV
 * launch per matrix.  Each Y_i equals
 * jllm_q4k_gemm(w_q4k[i], ...) within the matmul bound (the fp32
 * summation order of cut tiles follows the batch's split).
 * Errors: INVALID_ARG (also count outside 1..4), UNSUPPORTED_SHAPE,
 *         MISALIGNED, UNSUPPORTED_DTYPE, WORKSPACE, CUDA.
 */
jllm_status jllm_q4k_gemm_batch(const void* const* w_q4k, const void* x, void* const* y, jllm_dtype y_dt,
                                int64_t M, const int64_t* N, int64_t K, int count, void* ws,
                                size_t ws_bytes, jllm_stream_t stream);

/*
 * jllm_q4k_ffn_swiglu -- h = silu(X*Wg^T) * (X*Wu^T), the gate/up half of a
 * SwiGLU MLP in one pass over X (the README's "fused ... SwiGLU", Kernels
 * bullet).  silu(z) = z / (1 + e^-z).
 *   w_gate, w_up : two Q4_K matrices, each [N][K/256] blocks
 *   x     : [M][K] fp16
 *   h     : [M][N] fp16
 *   ws, ws_bytes : optional workspace, as for jllm_q4k_gemm
 * g and u are each accurate to the matmul bound above; h is silu(g)*u
 * evaluated in fp32 and rounded to fp16.
 * Errors: as jllm_q4k_gemm.
 */
jllm_status jllm_q4k_ffn_swiglu(const void* w_gate, const void* w_up, const void* x, void* h,
                                int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes,
                                jllm_stream_t stream);

/*
 * jllm_kv_encode_i8 / jllm_kv_decode_i8 -- the FP16 <-> INT8 KV cache codec
 * (the README's "FP16<->INT8 KV convert" kernel, Project layout, src/kernels/;
 * At a glance, KV cache bullet: "INT8 by default", "FP16-ULP-bounded drift").
 * The pages give no scale granularity or rounding; this library's rule: one
 * scale per vector of head_dim values (one head of one token), symmetric, a
 * power of two s = 2^e stored as fp16, e the smallest integer with
 * max|v| <= 127 * 2^e clamped to [-24, 9];
 *   encode: q = round-half-even(v / s) clamped to [-127, 127]
 *   decode: v' = q * s (exact in fp16)
 * so |v' - v| <= s/2 (<= s where the code saturates, max|v| > 65280), and
 * decode(encode(decode(encode(v)))) == decode(encode(v)) bit for bit: the
 * codec does not drift under repeated round trips.  Codes and scales are
 * bit-exact to that rule for finite inputs (non-finite values give
 * unspecified codes).
 *   kv      : [n_vectors][head_dim] fp16, 16-byte aligned
 *   codes   : [n_vectors][head_dim] int8, 16-byte aligned
 *   scales  : [n_vectors] fp16, 2-byte aligned
 *   head_dim: 64, 128 or 256
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
jllm_status jllm_kv_encode_i8(const void* kv, int8_t* codes, void* scales, int64_t n_vectors, int64_t head_dim,
                              jllm_stream_t stream);
jllm_status jllm_kv_decode_i8(const int8_t* codes, const void* scales, void* kv, int64_t n_vectors,
                              int64_t head_dim, jllm_stream_t stream);

/*
 * Workspace bytes that gemm/ffn_swiglu can use for this shape on the current
 * device (0 = the call takes none).  It depends on M, N and K only: a GEMM
 * that the few-token kernel takes ignores a workspace it is given, while
 * jllm_q4k_ffn_swiglu at the same M runs the tcgen05 kernel and can use it.
 * Passing ws = NULL is always allowed and only gives up the stream-K split.  A workspace that is given must be at
 * least this large, 256-byte aligned, and zero-filled before its first use;
 * every call that completes leaves it zero-filled where that matters, so it
 * can be reused by later calls, one call at a time (calls on different
 * streams need different workspaces).  After JLLM_ERR_DEVICE_TIMEOUT,
 * zero-fill it again.  Owned by the caller.
 */
size_t jllm_q4k_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Largest M that jllm_q4k_gemm sends to the CUDA-core GEMV kernel (which
 * handles up to 8 tokens per launch); larger M run the few-token or the
 * tcgen05 kernel (jllm_q4k_gemm).  The
 * default (1) is the measured crossover with the few-token kernel, which is
 * faster from two tokens; the environment variable JLLM_GEMV_MAX_M (0..8),
 * read once per process, overrides it.
 * jllm_q4k_ffn_swiglu uses the GEMV for M = 1 only.
 */
int jllm_q4k_gemv_max_m(void);

/*
 * Synchronise `stream`, then read and clear the device error words (current
 * device) that a kernel sets when one of its bounded waits runs out.  When a
 * tcgen05 GEMM timed out, the stream-K flags of the library's static
 * workspace (jllm_q4k_gemm_noalloc) are zeroed as well; a caller-owned
 * workspace must be zero-filled again by its owner.  Returns JLLM_OK,
 * JLLM_ERR_DEVICE_TIMEOUT or JLLM_ERR_CUDA.
 */
jllm_status jllm_get_device_error(jllm_stream_t stream);

/* Static, NUL-terminated name of a status code. */
const char* jllm_status_string(jllm_status status);

#ifdef __cplusplus
}
#endif

#endif /* JLLM_Q4K_H */

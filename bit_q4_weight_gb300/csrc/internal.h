// Internal launchers shared by the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "jllm_q4k.h"

namespace jllm {

struct DevInfo {
  int device = -1;
  int sm_count = 0;
  int major = 0, minor = 0;
  size_t smem_optin = 0;  // max dynamic shared memory per block
  bool pdl = true;        // launch GEMV kernels with programmatic dependent launch
  cudaError_t err = cudaSuccess;
};

// Properties of the current device (cached per device).
const DevInfo& device_info();

// out[N,K] = dequant(W); f16 selects fp16 output.
cudaError_t launch_dequant(const void* w, void* out, bool f16, int64_t N, int64_t K, cudaStream_t s);

// CUDA-core GEMV for M <= kMaxGemvTokens tokens.  w1 == nullptr:
// y[M][N] = x[M][K] W0^T, fp32 (y_f16: fp16).  w1 != nullptr (M = 1 only):
// y = fp16 [N] = silu(W0 x) * (W1 x).
constexpr int kMaxGemvTokens = 8;
cudaError_t launch_gemv(const void* w0, const void* w1, const void* x, void* y, int64_t N, int64_t K, int M,
                        bool y_f16, cudaStream_t s);

// Up to kMaxGemvBatch M = 1 GEMVs over the same x (and K) in one launch:
// y[i] = fp32 [N[i]] = W[i] x.
constexpr int kMaxGemvBatch = 8;
cudaError_t launch_gemv_batch(const void* const* w, void* const* y, const int64_t* N, int count, const void* x,
                              int64_t K, cudaStream_t s);

// launch_gemv_batch on x normalised in the prologue:
// xn = fp16(x * gamma / sqrt(mean(x^2) + eps)), gamma fp32 [K], one token.
cudaError_t launch_gemv_batch_rmsnorm(const void* const* w, void* const* y, const int64_t* N, int count,
                                      const void* x, const float* gamma, float eps, int64_t K, cudaStream_t s);

// The q/k/v GEMVs of an attention block in one launch (w, y: 3 matrices
// over the same x, M = 1, fp32 outputs) with a rotary epilogue on the first
// n_rope (1 or 2) matrices: heads of 128 rows, optional per-head RMSNorm
// (head_gamma[i] [128] or nullptr), rotation by pos * base^(-2j/128) of
// pairs (j, j + 64).  gamma != nullptr adds the RMSNorm prologue on x.
// Every N[i] must be a multiple of 128.
cudaError_t launch_gemv_qkv_rope(const void* const* w, void* const* y, const int64_t* N, int n_rope,
                                 const float* const* head_gamma, float head_eps, int pos, double rope_base,
                                 const void* x, const float* gamma, float eps, int64_t K, cudaStream_t s);

// A sequence of one-token GEMV steps in one persistent cooperative launch
// (jllm_q4k_gemv_chain): step s+1 reads x only after every y of step s is
// written.  sync: n_steps + 1 zeroed words, left zeroed by a launch that
// completes.  At most kChainMaxSteps steps of kChainMaxMats matrices, K at
// most kChainMaxBlocks * 256.
constexpr int kChainMaxSteps = 256;
constexpr int kChainMaxMats = 4;
constexpr int kChainMaxBlocks = 48;
cudaError_t launch_gemv_chain(const jllm_gemv_step* steps, int n_steps, uint32_t* sync, cudaStream_t s);

// TMA + tcgen05 GEMM for any M >= 1.  w1 != nullptr selects the SwiGLU
// epilogue (y = fp16 h).  ws (nullptr allowed) of at least
// gemm_workspace_bytes() zero-initialised bytes enables the stream-K split.
// Returns cudaErrorInvalidValue for unsupported shapes.
cudaError_t launch_gemm_tc(const void* w0, const void* w1, const void* x, void* y, bool y_f16, int64_t M,
                           int64_t N, int64_t K, void* ws, size_t ws_bytes, cudaStream_t s);

// Up to kMaxGemmBatch tcgen05 GEMMs over the same x (and K) in one
// persistent launch: y[b] = [M][N[b]] = x W[b]^T, fp32 (y_f16: fp16).
constexpr int kMaxGemmBatch = 4;
cudaError_t launch_gemm_tc_batch(const void* const* w, const int64_t* N, int count, const void* x, void* const* y,
                                 bool y_f16, int64_t M, int64_t K, void* ws, size_t ws_bytes, cudaStream_t s);

// Warp-level tensor-core GEMM for a few tokens (gemm_mma.cu): y[b] = [M][N[b]]
// = x W[b]^T for 1 <= M <= kGemmMmaMaxM, up to kMaxGemmBatch matrices over
// the same x (fp32 out, y_f16: fp16).  No workspace: K is split over a
// thread-block cluster.  gemm_mma_takes() says whether the C ABI sends a call
// above the GEMV threshold to it (else the tcgen05 GEMM).
constexpr int kGemmMmaMaxM = 40;
bool gemm_mma_takes(int64_t M, const int64_t* N, int count);
cudaError_t launch_gemm_mma(const void* const* w, const int64_t* N, int count, const void* x, void* const* y,
                            bool y_f16, int64_t M, int64_t K, cudaStream_t s);

// Tensor maps shared by the TMA kernels (cached per device and buffer):
// x [M][K] fp16 as 64-wide boxes of box_tokens rows with the 128-byte swizzle;
// W [N][K/256] Q4_K blocks as a byte view, one super-block of box_rows rows per box.
cudaError_t tma_map_x(const void* x, int64_t M, int64_t K, int box_tokens, CUtensorMap* map);
cudaError_t tma_map_w(const void* w, int64_t N, int64_t K, int box_rows, CUtensorMap* map);

// FP16 <-> INT8 KV codec over n_vec vectors of dim (64, 128 or 256) values:
// codes [n_vec][dim] int8, one fp16 power-of-two scale per vector.
cudaError_t launch_kv_encode(const void* kv, int8_t* codes, void* scales, int64_t n_vec, int dim, cudaStream_t s);
cudaError_t launch_kv_decode(const int8_t* codes, const void* scales, void* kv, int64_t n_vec, int dim, cudaStream_t s);

// Workspace of the stream-K split on the current device: one 128 KiB fp32
// partial slot and one flag word per SM (0 when the device is unusable).
size_t gemm_workspace_bytes();

// The library's own static device workspace (address on the current device,
// looked up once per device, and its size).
cudaError_t gemm_static_workspace(void** ptr, size_t* bytes);

// Zero the stream-K flag words of the static workspace on the current device
// (enqueued on s, then s is synchronised); a no-op if it was never used.
cudaError_t gemm_static_workspace_reset(cudaStream_t s);

#ifdef JLLM_FAULT_INJECTION
// Test builds only: make one bounded wait of the next launches run out.
cudaError_t fault_injection_set_gemm(int skip_x);
cudaError_t fault_injection_set_gemv(int skip_w);
cudaError_t fault_injection_set_chain(int skip);
cudaError_t fault_injection_set_mma(int skip);
#endif

// Read and clear the device error word of the tcgen05 kernels (after
// synchronising the stream), of the GEMV kernels and of the GEMV chain.
cudaError_t read_clear_gemm_error(uint32_t* bits, cudaStream_t s);
cudaError_t read_clear_gemv_error(uint32_t* bits);
cudaError_t read_clear_chain_error(uint32_t* bits);
cudaError_t read_clear_mma_error(uint32_t* bits);

}  // namespace jllm

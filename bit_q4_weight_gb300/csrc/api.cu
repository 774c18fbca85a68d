// C ABI of the Q4_K library (include/jllm_q4k.h): argument checks, the
// M-threshold dispatch between the GEMV and the tcgen05 GEMM, and status
// mapping.  Nothing here allocates device memory.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>

#include "../../include/jllm_q4k.h"
#include "internal.h"

namespace jllm {

namespace {
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
}  // namespace

const DevInfo& device_info() {
  static thread_local DevInfo bad;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    bad.err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return bad;
  }
  std::call_once(g_dev_once[dev], [dev]() {
    DevInfo& d = g_dev[dev];
    d.device = dev;
    cudaError_t err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    int optin = 0;
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.smem_optin = (size_t)optin;
    const char* env = getenv("JLLM_PDL");
    d.pdl = !(env && env[0] == '0');
    d.err = err;
  });
  return g_dev[dev];
}

}  // namespace jllm

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The kernels index rows and blocks with 32-bit integers.
constexpr int64_t kMaxRows = (int64_t)1 << 30;
constexpr int64_t kMaxK = (int64_t)1 << 24;

jllm_status check_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1) return JLLM_ERR_INVALID_ARG;
  if (K < 256 || K % 256 != 0) return JLLM_ERR_UNSUPPORTED_SHAPE;
  if (M > kMaxRows || N > kMaxRows || K > kMaxK) return JLLM_ERR_UNSUPPORTED_SHAPE;
  return JLLM_OK;
}

// The workspace is optional: NULL runs without it; a given one must be
// large enough and aligned.
jllm_status check_workspace(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || need == 0) return JLLM_OK;
  if (ws_bytes < need || ((uintptr_t)ws & 255u) != 0) return JLLM_ERR_WORKSPACE;
  return JLLM_OK;
}

jllm_status check_device() {
  const jllm::DevInfo& d = jllm::device_info();
  if (d.err != cudaSuccess) return JLLM_ERR_CUDA;
  if (d.major != 10 || d.minor != 3) return JLLM_ERR_NO_DEVICE;
  return JLLM_OK;
}

jllm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? JLLM_OK : JLLM_ERR_CUDA; }

// Largest M sent to the CUDA-core GEMV (the few-token and tcgen05 GEMMs take the
// rest).  1 from the measured crossover with the few-token GEMM: from two tokens
// that kernel is faster on every layer shape (2560->6144, 4096->2560,
// 2560->19456, 9728->2560: 1.0-2.4x at M = 2..4).  JLLM_GEMV_MAX_M overrides it
// within 0..kMaxGemvTokens.
int g_gemv_max_m = 1;
std::once_flag g_thresh_once;

int gemv_max_m() {
  std::call_once(g_thresh_once, []() {
    const char* env = getenv("JLLM_GEMV_MAX_M");
    if (env) {
      const long v = strtol(env, nullptr, 10);
      if (v >= 0 && v <= jllm::kMaxGemvTokens) g_gemv_max_m = (int)v;
    }
  });
  return g_gemv_max_m;
}

}  // namespace

extern "C" {

const char* jllm_status_string(jllm_status status) {
  switch (status) {
    case JLLM_OK: return "JLLM_OK";
    case JLLM_ERR_INVALID_ARG: return "JLLM_ERR_INVALID_ARG";
    case JLLM_ERR_UNSUPPORTED_SHAPE: return "JLLM_ERR_UNSUPPORTED_SHAPE";
    case JLLM_ERR_MISALIGNED: return "JLLM_ERR_MISALIGNED";
    case JLLM_ERR_UNSUPPORTED_DTYPE: return "JLLM_ERR_UNSUPPORTED_DTYPE";
    case JLLM_ERR_WORKSPACE: return "JLLM_ERR_WORKSPACE";
    case JLLM_ERR_CUDA: return "JLLM_ERR_CUDA";
    case JLLM_ERR_DEVICE_TIMEOUT: return "JLLM_ERR_DEVICE_TIMEOUT";
    case JLLM_ERR_NO_DEVICE: return "JLLM_ERR_NO_DEVICE";
  }
  return "JLLM_ERR_UNKNOWN";
}

int jllm_q4k_gemv_max_m(void) { return gemv_max_m(); }

size_t jllm_q4k_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (check_shape(M, N, K) != JLLM_OK || M <= gemv_max_m()) return 0;
  return jllm::gemm_workspace_bytes();
}

jllm_status jllm_q4k_dequant(const void* w_q4k, void* out, jllm_dtype out_dt, int64_t N, int64_t K,
                             jllm_stream_t stream) {
  if (!w_q4k || !out) return JLLM_ERR_INVALID_ARG;
  jllm_status st = check_shape(1, N, K);
  if (st != JLLM_OK) return st;
  if (out_dt != JLLM_F32 && out_dt != JLLM_F16) return JLLM_ERR_UNSUPPORTED_DTYPE;
  if (!aligned16(w_q4k) || !aligned16(out)) return JLLM_ERR_MISALIGNED;
  if ((st = check_device()) != JLLM_OK) return st;
  return from_cuda(jllm::launch_dequant(w_q4k, out, out_dt == JLLM_F16, N, K, (cudaStream_t)stream));
}

jllm_status jllm_q4k_gemv(const void* w_q4k, const void* x, float* y, int64_t N, int64_t K, void* ws,
                          size_t ws_bytes, jllm_stream_t stream) {
  if (!w_q4k || !x || !y) return JLLM_ERR_INVALID_ARG;
  jllm_status st = check_shape(1, N, K);
  if (st != JLLM_OK) return st;
  if (!aligned16(w_q4k) || !aligned16(x) || !aligned16(y)) return JLLM_ERR_MISALIGNED;
  if ((st = check_workspace(ws, ws_bytes, jllm_q4k_workspace_bytes(1, N, K))) != JLLM_OK) return st;
  if ((st = check_device()) != JLLM_OK) return st;
  return from_cuda(jllm::launch_gemv(w_q4k, nullptr, x, y, N, K, 1, false, (cudaStream_t)stream));
}

jllm_status jllm_q4k_gemv_batch(const void* const* w_q4k, float* const* y, const int64_t* N, int count,
                                const void* x, int64_t K, jllm_stream_t stream) {
  if (!w_q4k || !y || !N || !x) return JLLM_ERR_INVALID_ARG;
  if (count < 1 || count > jllm::kMaxGemvBatch) return JLLM_ERR_INVALID_ARG;
  if (!aligned16(x)) return JLLM_ERR_MISALIGNED;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) {
    if (!w_q4k[i] || !y[i]) return JLLM_ERR_INVALID_ARG;
    jllm_status st = check_shape(1, N[i], K);
    if (st != JLLM_OK) return st;
    if (!aligned16(w_q4k[i]) || !aligned16(y[i])) return JLLM_ERR_MISALIGNED;
    total += N[i];
  }
  if (total > kMaxRows) return JLLM_ERR_UNSUPPORTED_SHAPE;
  jllm_status st = check_device();
  if (st != JLLM_OK) return st;
  return from_cuda(jllm::launch_gemv_batch(w_q4k, reinterpret_cast<void* const*>(y), N, count, x, K,
                                           (cudaStream_t)stream));
}

jllm_status jllm_q4k_gemv_rmsnorm_batch(const void* const* w_q4k, float* const* y, const int64_t* N, int count,
                                        const void* x, const float* gamma, float eps, int64_t K,
                                        jllm_stream_t stream) {
  if (!w_q4k || !y || !N || !x || !gamma) return JLLM_ERR_INVALID_ARG;
  if (count < 1 || count > jllm::kMaxGemvBatch) return JLLM_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || eps > 1.f) return JLLM_ERR_INVALID_ARG;  // also rejects NaN
  if (!aligned16(x) || !aligned16(gamma)) return JLLM_ERR_MISALIGNED;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) {
    if (!w_q4k[i] || !y[i]) return JLLM_ERR_INVALID_ARG;
    jllm_status st = check_shape(1, N[i], K);
    if (st != JLLM_OK) return st;
    if (!aligned16(w_q4k[i]) || !aligned16(y[i])) return JLLM_ERR_MISALIGNED;
    total += N[i];
  }
  if (total > kMaxRows) return JLLM_ERR_UNSUPPORTED_SHAPE;
  jllm_status st = check_device();
  if (st != JLLM_OK) return st;
  return from_cuda(jllm::launch_gemv_batch_rmsnorm(w_q4k, reinterpret_cast<void* const*>(y), N, count, x, gamma,
                                                   eps, K, (cudaStream_t)stream));
}

jllm_status jllm_q4k_gemv_chain(const jllm_gemv_step* steps, int n_steps, uint32_t* sync, jllm_stream_t stream) {
  if (!steps || !sync) return JLLM_ERR_INVALID_ARG;
  if (n_steps < 1 || n_steps > JLLM_CHAIN_MAX_STEPS) return JLLM_ERR_INVALID_ARG;
  if (((uintptr_t)sync & 3u) != 0) return JLLM_ERR_MISALIGNED;
  for (int s = 0; s < n_steps; ++s) {
    const jllm_gemv_step& d = steps[s];
    if (!d.x || d.count < 1 || d.count > JLLM_CHAIN_MAX_MATS || (d.y_f16 != 0 && d.y_f16 != 1))
      return JLLM_ERR_INVALID_ARG;
    if (d.K <= 0 || d.K % 256 || d.K > JLLM_CHAIN_MAX_K) return JLLM_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(d.x)) return JLLM_ERR_MISALIGNED;
    int64_t total = 0;
    for (int i = 0; i < d.count; ++i) {
      if (d.N[i] < 0) return JLLM_ERR_INVALID_ARG;
      if (d.N[i] == 0) continue;
      if (!d.w_q4k[i] || !d.y[i]) return JLLM_ERR_INVALID_ARG;
      if (!aligned16(d.w_q4k[i]) || !aligned16(d.y[i])) return JLLM_ERR_MISALIGNED;
      total += d.N[i];
    }
    if (total > kMaxRows) return JLLM_ERR_UNSUPPORTED_SHAPE;
  }
  jllm_status st = check_device();
  if (st != JLLM_OK) return st;
  return from_cuda(jllm::launch_gemv_chain(steps, n_steps, sync, (cudaStream_t)stream));
}

size_t jllm_q4k_gemv_chain_sync_bytes(int n_steps) {
  return (n_steps < 1 || n_steps > JLLM_CHAIN_MAX_STEPS) ? 0 : sizeof(uint32_t) * (size_t)(n_steps + 1);
}

jllm_status jllm_q4k_gemv_qkv_rope(const void* const* w_q4k, float* const* y, int64_t n_q_heads,
                                   int64_t n_kv_heads, const void* x, int64_t K, const float* gamma, float eps,
                                   const float* q_gamma, const float* k_gamma, float head_eps, int64_t pos,
                                   float rope_base, jllm_stream_t stream) {
  if (!w_q4k || !y || !x) return JLLM_ERR_INVALID_ARG;
  if (n_q_heads < 1 || n_kv_heads < 1) return JLLM_ERR_INVALID_ARG;
  if (gamma && (!(eps >= 0.f) || eps > 1.f)) return JLLM_ERR_INVALID_ARG;
  if ((q_gamma || k_gamma) && (!(head_eps >= 0.f) || head_eps > 1.f)) return JLLM_ERR_INVALID_ARG;
  if (!(rope_base > 0.f) || !isfinite(rope_base)) return JLLM_ERR_INVALID_ARG;
  if (pos < INT32_MIN || pos > INT32_MAX) return JLLM_ERR_INVALID_ARG;
  if (!aligned16(x) || (gamma && !aligned16(gamma)) || (q_gamma && !aligned16(q_gamma)) ||
      (k_gamma && !aligned16(k_gamma)))
    return JLLM_ERR_MISALIGNED;
  const int64_t head = 128;
  if (n_q_heads > kMaxRows / head || n_kv_heads > kMaxRows / head) return JLLM_ERR_UNSUPPORTED_SHAPE;
  const int64_t N[3] = {n_q_heads * head, n_kv_heads * head, n_kv_heads * head};
  for (int i = 0; i < 3; ++i) {
    if (!w_q4k[i] || !y[i]) return JLLM_ERR_INVALID_ARG;
    jllm_status st = check_shape(1, N[i], K);
    if (st != JLLM_OK) return st;
    if (!aligned16(w_q4k[i]) || !aligned16(y[i])) return JLLM_ERR_MISALIGNED;
  }
  if (N[0] + N[1] + N[2] > kMaxRows) return JLLM_ERR_UNSUPPORTED_SHAPE;
  jllm_status st = check_device();
  if (st != JLLM_OK) return st;
  const float* hg[2] = {q_gamma, k_gamma};
  return from_cuda(jllm::launch_gemv_qkv_rope(w_q4k, reinterpret_cast<void* const*>(y), N, 2, hg, head_eps, (int)pos,
                                              (double)rope_base, x, gamma, eps, K, (cudaStream_t)stream));
}

jllm_status jllm_q4k_gemm(const void* w_q4k, const void* x, void* y, jllm_dtype y_dt, int64_t M, int64_t N,
                          int64_t K, void* ws, size_t ws_bytes, jllm_stream_t stream) {
  if (!w_q4k || !x || !y) return JLLM_ERR_INVALID_ARG;
  jllm_status st = check_shape(M, N, K);
  if (st != JLLM_OK) return st;
  if (y_dt != JLLM_F32 && y_dt != JLLM_F16) return JLLM_ERR_UNSUPPORTED_DTYPE;
  if (!aligned16(w_q4k) || !aligned16(x) || !aligned16(y)) return JLLM_ERR_MISALIGNED;
  if ((st = check_workspace(ws, ws_bytes, jllm_q4k_workspace_bytes(M, N, K))) != JLLM_OK) return st;
  if ((st = check_device()) != JLLM_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (M <= gemv_max_m())
    return from_cuda(jllm::launch_gemv(w_q4k, nullptr, x, y, N, K, (int)M, y_dt == JLLM_F16, s));
  if (jllm::gemm_mma_takes(M, &N, 1))
    return from_cuda(jllm::launch_gemm_mma(&w_q4k, &N, 1, x, &y, y_dt == JLLM_F16, M, K, s));
  return from_cuda(jllm::launch_gemm_tc(w_q4k, nullptr, x, y, y_dt == JLLM_F16, M, N, K, ws, ws_bytes, s));
}

jllm_status jllm_q4k_gemm_noalloc(const void* w_q4k, const void* x, void* y, jllm_dtype y_dt, int64_t M,
                                  int64_t N, int64_t K, jllm_stream_t stream) {
  if (!w_q4k || !x || !y) return JLLM_ERR_INVALID_ARG;
  jllm_status st = check_shape(M, N, K);
  if (st != JLLM_OK) return st;
  if (y_dt != JLLM_F32 && y_dt != JLLM_F16) return JLLM_ERR_UNSUPPORTED_DTYPE;
  if (!aligned16(w_q4k) || !aligned16(x) || !aligned16(y)) return JLLM_ERR_MISALIGNED;
  if ((st = check_device()) != JLLM_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (M <= gemv_max_m())
    return from_cuda(jllm::launch_gemv(w_q4k, nullptr, x, y, N, K, (int)M, y_dt == JLLM_F16, s));
  if (jllm::gemm_mma_takes(M, &N, 1))
    return from_cuda(jllm::launch_gemm_mma(&w_q4k, &N, 1, x, &y, y_dt == JLLM_F16, M, K, s));
  void* ws = nullptr;
  size_t ws_bytes = 0;
  cudaError_t e = jllm::gemm_static_workspace(&ws, &ws_bytes);
  if (e != cudaSuccess) return JLLM_ERR_CUDA;
  if (ws_bytes < jllm_q4k_workspace_bytes(M, N, K)) return JLLM_ERR_WORKSPACE;  // more SMs than it was sized for
  return from_cuda(jllm::launch_gemm_tc(w_q4k, nullptr, x, y, y_dt == JLLM_F16, M, N, K, ws, ws_bytes, s));
}

jllm_status jllm_q4k_gemm_batch(const void* const* w_q4k, const void* x, void* const* y, jllm_dtype y_dt, int64_t M,
                                const int64_t* N, int64_t K, int count, void* ws, size_t ws_bytes,
                                jllm_stream_t stream) {
  if (!w_q4k || !x || !y || !N) return JLLM_ERR_INVALID_ARG;
  if (count < 1 || count > jllm::kMaxGemmBatch) return JLLM_ERR_INVALID_ARG;
  if (y_dt != JLLM_F32 && y_dt != JLLM_F16) return JLLM_ERR_UNSUPPORTED_DTYPE;
  if (!aligned16(x)) return JLLM_ERR_MISALIGNED;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) {
    if (!w_q4k[i] || !y[i]) return JLLM_ERR_INVALID_ARG;
    jllm_status st = check_shape(M, N[i], K);
    if (st != JLLM_OK) return st;
    if (!aligned16(w_q4k[i]) || !aligned16(y[i])) return JLLM_ERR_MISALIGNED;
    total += N[i];
  }
  if (total > kMaxRows) return JLLM_ERR_UNSUPPORTED_SHAPE;
  jllm_status st = check_workspace(ws, ws_bytes, jllm_q4k_workspace_bytes(M, total, K));
  if (st != JLLM_OK) return st;
  if ((st = check_device()) != JLLM_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const bool f16 = y_dt == JLLM_F16;
  if (M <= gemv_max_m()) {
    for (int i = 0; i < count; ++i) {
      st = from_cuda(jllm::launch_gemv(w_q4k[i], nullptr, x, y[i], N[i], K, (int)M, f16, s));
      if (st != JLLM_OK) return st;
    }
    return JLLM_OK;
  }
  if (jllm::gemm_mma_takes(M, N, count)) return from_cuda(jllm::launch_gemm_mma(w_q4k, N, count, x, y, f16, M, K, s));
  return from_cuda(jllm::launch_gemm_tc_batch(w_q4k, N, count, x, y, f16, M, K, ws, ws_bytes, s));
}

jllm_status jllm_q4k_ffn_swiglu(const void* w_gate, const void* w_up, const void* x, void* h, int64_t M,
                                int64_t N, int64_t K, void* ws, size_t ws_bytes, jllm_stream_t stream) {
  if (!w_gate || !w_up || !x || !h) return JLLM_ERR_INVALID_ARG;
  jllm_status st = check_shape(M, N, K);
  if (st != JLLM_OK) return st;
  if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(x) || !aligned16(h)) return JLLM_ERR_MISALIGNED;
  if ((st = check_workspace(ws, ws_bytes, jllm_q4k_workspace_bytes(M, N, K))) != JLLM_OK) return st;
  if ((st = check_device()) != JLLM_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (M == 1 && gemv_max_m() >= 1) return from_cuda(jllm::launch_gemv(w_gate, w_up, x, h, N, K, 1, true, s));
  return from_cuda(jllm::launch_gemm_tc(w_gate, w_up, x, h, true, M, N, K, ws, ws_bytes, s));
}

static jllm_status check_kv(const void* a, const void* b, const void* scales, int64_t n_vectors, int64_t head_dim) {
  if (!a || !b || !scales) return JLLM_ERR_INVALID_ARG;
  if (n_vectors < 1) return JLLM_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return JLLM_ERR_UNSUPPORTED_SHAPE;
  if (n_vectors > ((int64_t)1 << 40) / head_dim) return JLLM_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(b) || ((uintptr_t)scales & 1u)) return JLLM_ERR_MISALIGNED;
  return check_device();
}

jllm_status jllm_kv_encode_i8(const void* kv, int8_t* codes, void* scales, int64_t n_vectors, int64_t head_dim,
                              jllm_stream_t stream) {
  jllm_status st = check_kv(kv, codes, scales, n_vectors, head_dim);
  if (st != JLLM_OK) return st;
  return from_cuda(jllm::launch_kv_encode(kv, codes, scales, n_vectors, (int)head_dim, (cudaStream_t)stream));
}

jllm_status jllm_kv_decode_i8(const int8_t* codes, const void* scales, void* kv, int64_t n_vectors, int64_t head_dim,
                              jllm_stream_t stream) {
  jllm_status st = check_kv(codes, kv, scales, n_vectors, head_dim);
  if (st != JLLM_OK) return st;
  return from_cuda(jllm::launch_kv_decode(codes, scales, kv, n_vectors, (int)head_dim, (cudaStream_t)stream));
}

jllm_status jllm_get_device_error(jllm_stream_t stream) {
  uint32_t a = 0, b = 0, c = 0, d = 0;
  cudaError_t e = jllm::read_clear_gemm_error(&a, (cudaStream_t)stream);
  if (e == cudaSuccess) e = jllm::read_clear_gemv_error(&b);
  if (e == cudaSuccess) e = jllm::read_clear_chain_error(&c);
  if (e == cudaSuccess) e = jllm::read_clear_mma_error(&d);
  // A tcgen05 kernel that gave up may have left stream-K flags set in the
  // library's static workspace: clear them before anyone calls again.
  if (e == cudaSuccess && a) e = jllm::gemm_static_workspace_reset((cudaStream_t)stream);
  if (e != cudaSuccess) return JLLM_ERR_CUDA;
  return (a | b | c | d) ? JLLM_ERR_DEVICE_TIMEOUT : JLLM_OK;
}

#ifdef JLLM_FAULT_INJECTION
// Test builds only (not declared in the public header): gemm_skip_x makes CTA
// 0 of the next tcgen05 GEMMs skip its first X copy, gemv_skip_w makes warp 0
// of CTA 0 of the next GEMVs skip its weight copy; 0 clears either.
jllm_status jllm_test_fault_injection(int gemm_skip_x, int gemv_skip_w) {
  cudaError_t e = jllm::fault_injection_set_gemm(gemm_skip_x);
  if (e == cudaSuccess) e = jllm::fault_injection_set_gemv(gemv_skip_w);
  return from_cuda(e);
}

// Test builds only: skip != 0 makes the producer of CTA 0 of the next GEMV
// chains skip its first weight copy; 0 clears it.
jllm_status jllm_test_fault_injection_chain(int skip) { return from_cuda(jllm::fault_injection_set_chain(skip)); }

// Test builds only: skip != 0 makes CTA 0 of the next few-token (mma.sync)
// GEMMs skip its first x copies; 0 clears it.
jllm_status jllm_test_fault_injection_mma(int skip) { return from_cuda(jllm::fault_injection_set_mma(skip)); }
#endif

}  // extern "C"

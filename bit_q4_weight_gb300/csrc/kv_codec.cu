// FP16 <-> INT8 KV cache codec: the "FP16<->INT8 KV convert" kernel of the
// genie-ai-runtime README (Project layout, src/kernels/; At a glance, KV cache
// bullet: INT8 by default, "FP16-ULP-bounded drift").
//
// One scale per vector of D fp16 values (one head of one token), symmetric,
// the scale a power of two s = 2^e stored as fp16: e is the smallest integer
// with max|v| <= 127 * 2^e, clamped to [-24, 9]; codes are
// round-half-even(v / 2^e) clamped to [-127, 127]; decode is q * 2^e, which is
// exact in fp16, so a second round trip reproduces the codes and the values.
//
// Both directions are HBM-bound streams.  A vector is handled by D/8 lanes of
// a warp, each moving 16 bytes of fp16 (8 values) and 8 code bytes; the
// vector's max |v| is a shuffle reduction within those lanes.  Each thread
// keeps UNROLL vectors' loads in flight before it computes, over a grid of a
// few CTAs per SM that strides through the vectors.
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace jllm {
namespace {

constexpr int KV_THREADS = 256;
constexpr int KV_UNROLL = 4;

// 2^e as fp32, for the exponents used here (normal range).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Exponent e of the scale for a vector whose largest magnitude is a (finite,
// >= 0, an fp16 value, so a normal fp32): with a = f * 2^E, f in [0.5, 1), e
// is E - 7 or E - 6 (127 * 2^(E-7) < 2^E and 127 * 2^(E-6) >= 2^E > a); one
// exact comparison picks it.
__device__ __forceinline__ int kv_exponent(float a) {
  if (a == 0.f) return -24;
  const int E = ((__float_as_int(a) >> 23) & 0xff) - 126;
  int e = E - 7;
  if (a > 127.f * pow2f(e)) ++e;
  return e < -24 ? -24 : (e > 9 ? 9 : e);
}

__device__ __forceinline__ uint32_t pack4_i8(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) | ((uint32_t)(d & 0xff) << 24);
}

__device__ __forceinline__ int code_of(float v, float inv) {
  int q = __float2int_rn(v * inv);  // v * 2^-e is exact; round half to even
  return q > 127 ? 127 : (q < -127 ? -127 : q);
}

// L = lanes per vector (D / 8).
template <int L>
__global__ void __launch_bounds__(KV_THREADS, 5) kv_encode_kernel(const uint4* __restrict__ kv, uint2* __restrict__ codes,
                                                               __half* __restrict__ scales, int64_t n_vec) {
  constexpr int VPW = 32 / L;  // vectors per warp and pass
  const int lane = threadIdx.x & 31, sub = lane % L;
  const int64_t warps = (int64_t)gridDim.x * (KV_THREADS / 32);
  const int64_t gw = (int64_t)blockIdx.x * (KV_THREADS / 32) + (threadIdx.x >> 5);
  const int64_t stride = warps * VPW;
  // The loop bound is the warp's first vector, so every lane of a warp runs the
  // same iterations (the shuffles below need all 32); lanes past the end are
  // predicated off.
  for (int64_t wbase = gw * VPW; wbase < n_vec; wbase += stride * KV_UNROLL) {
    const int64_t base = wbase + lane / L;
    uint4 u[KV_UNROLL];
#pragma unroll
    for (int j = 0; j < KV_UNROLL; ++j) {
      const int64_t v = base + (int64_t)j * stride;
      u[j] = v < n_vec ? ldg_stream(kv + v * L + sub) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < KV_UNROLL; ++j) {
      const int64_t v = base + (int64_t)j * stride;
      // largest |v| of the lane's 8 values: fp16 magnitudes compare as integers
      const uint32_t w[4] = {u[j].x & 0x7fff7fffu, u[j].y & 0x7fff7fffu, u[j].z & 0x7fff7fffu, u[j].w & 0x7fff7fffu};
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0xffffu, w[i] >> 16));
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int e = kv_exponent(__half2float(__ushort_as_half((unsigned short)m)));
      if (v < n_vec) {
        uint2 out;
        if (e >= -14) {
          // fp16 pairs: fma(v, 2^-e, 1536) is v / 2^e + 1536 rounded once to the fp16 grid of
          // [1024, 2048), whose step is 1: round half to even of v / 2^e, plus 1536.  The
          // bits are then 0x6600 + q, so the low byte is q as a two's-complement int8.
          // |v / 2^e| <= 127 except when e is clamped at 9 (max |v| > 65280): clamp there.
          const uint32_t inv = (uint32_t)(15 - e) << 10;  // fp16 2^-e
          const uint32_t inv2 = inv | (inv << 16);
          uint32_t r[4];
          const uint32_t w[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[i]) : "r"(w[i]), "r"(inv2), "r"(0x66006600u));
            if (e == 9) {  // 1536 -/+ 127 = 0x6581 / 0x667F
              asm("max.f16x2 %0, %0, %1;" : "+r"(r[i]) : "r"(0x65816581u));
              asm("min.f16x2 %0, %0, %1;" : "+r"(r[i]) : "r"(0x667F667Fu));
            }
          }
          out.x = __byte_perm(r[0], r[1], 0x6420);  // low bytes of the four halves
          out.y = __byte_perm(r[2], r[3], 0x6420);
        } else {
          const float inv = pow2f(-e);
          const __half2* h = reinterpret_cast<const __half2*>(&u[j]);
          float2 f0 = __half22float2(h[0]), f1 = __half22float2(h[1]), f2 = __half22float2(h[2]), f3 = __half22float2(h[3]);
          out.x = pack4_i8(code_of(f0.x, inv), code_of(f0.y, inv), code_of(f1.x, inv), code_of(f1.y, inv));
          out.y = pack4_i8(code_of(f2.x, inv), code_of(f2.y, inv), code_of(f3.x, inv), code_of(f3.y, inv));
        }
        codes[v * L + sub] = out;
        if (sub == 0) scales[v] = __float2half_rn(pow2f(e));
      }
    }
  }
}

template <int L>
__global__ void __launch_bounds__(KV_THREADS) kv_decode_kernel(const uint2* __restrict__ codes,
                                                               const __half* __restrict__ scales, uint4* __restrict__ kv,
                                                               int64_t n_vec) {
  constexpr int VPW = 32 / L;
  const int lane = threadIdx.x & 31, sub = lane % L;
  const int64_t warps = (int64_t)gridDim.x * (KV_THREADS / 32);
  const int64_t gw = (int64_t)blockIdx.x * (KV_THREADS / 32) + (threadIdx.x >> 5);
  const int64_t stride = warps * VPW;
  for (int64_t wbase = gw * VPW; wbase < n_vec; wbase += stride * KV_UNROLL) {
    const int64_t base = wbase + lane / L;
    uint2 c[KV_UNROLL];
    float s[KV_UNROLL];
#pragma unroll
    for (int j = 0; j < KV_UNROLL; ++j) {
      const int64_t v = base + (int64_t)j * stride;
      if (v < n_vec) {
        uint2 t;
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(t.x), "=r"(t.y) : "l"(codes + v * L + sub));
        c[j] = t;
        s[j] = __half2float(scales[v]);
      } else {
        c[j] = make_uint2(0u, 0u);
        s[j] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < KV_UNROLL; ++j) {
      const int64_t v = base + (int64_t)j * stride;
      if (v >= n_vec) continue;
      const int8_t* b = reinterpret_cast<const int8_t*>(&c[j]);
      __half2 h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)  // q * 2^e: exact in fp32 and in fp16
        h[i] = __floats2half2_rn((float)b[2 * i] * s[j], (float)b[2 * i + 1] * s[j]);
      kv[v * L + sub] = *reinterpret_cast<const uint4*>(h);
    }
  }
}

// One wave: as many CTAs as can be resident at once (the kernel's occupancy,
// queried once per kernel and device), fewer when the vectors do not need them;
// the grid-stride loop covers the rest.  A grid of several partial waves would
// leave the last one running with part of the SMs' warps.
template <typename Kernel>
int kv_grid(Kernel kern, int which, int64_t n_vec, int L) {
  const DevInfo& dev = device_info();
  static std::atomic<int> resident[2][3][64];  // (encode/decode, L = 8/16/32, device)
  const int li = L == 8 ? 0 : (L == 16 ? 1 : 2);
  const int d = dev.device >= 0 && dev.device < 64 ? dev.device : 0;
  int per_sm = resident[which][li][d].load();
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, KV_THREADS, 0) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    cudaGetLastError();
    resident[which][li][d].store(per_sm);
  }
  const int64_t per_cta = (int64_t)(KV_THREADS / 32) * (32 / L) * KV_UNROLL;
  const int64_t want = (n_vec + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)dev.sm_count * per_sm;
  return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace

cudaError_t launch_kv_encode(const void* kv, int8_t* codes, void* scales, int64_t n_vec, int dim, cudaStream_t s) {
  const int L = dim / 8;
  const uint4* in = static_cast<const uint4*>(kv);
  uint2* out = reinterpret_cast<uint2*>(codes);
  __half* sc = static_cast<__half*>(scales);
  switch (L) {
    case 8: kv_encode_kernel<8><<<kv_grid(kv_encode_kernel<8>, 0, n_vec, L), KV_THREADS, 0, s>>>(in, out, sc, n_vec); break;
    case 16: kv_encode_kernel<16><<<kv_grid(kv_encode_kernel<16>, 0, n_vec, L), KV_THREADS, 0, s>>>(in, out, sc, n_vec); break;
    case 32: kv_encode_kernel<32><<<kv_grid(kv_encode_kernel<32>, 0, n_vec, L), KV_THREADS, 0, s>>>(in, out, sc, n_vec); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_kv_decode(const int8_t* codes, const void* scales, void* kv, int64_t n_vec, int dim, cudaStream_t s) {
  const int L = dim / 8;
  const uint2* in = reinterpret_cast<const uint2*>(codes);
  const __half* sc = static_cast<const __half*>(scales);
  uint4* out = static_cast<uint4*>(kv);
  switch (L) {
    case 8: kv_decode_kernel<8><<<kv_grid(kv_decode_kernel<8>, 1, n_vec, L), KV_THREADS, 0, s>>>(in, sc, out, n_vec); break;
    case 16: kv_decode_kernel<16><<<kv_grid(kv_decode_kernel<16>, 1, n_vec, L), KV_THREADS, 0, s>>>(in, sc, out, n_vec); break;
    case 32: kv_decode_kernel<32><<<kv_grid(kv_decode_kernel<32>, 1, n_vec, L), KV_THREADS, 0, s>>>(in, sc, out, n_vec); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace jllm

// Q4_K -> fp32 / fp16 dequantisation of a whole weight matrix.
//
// One warp per 144-byte super-block (grid-stride over blocks); lane l makes
// weights 8l..8l+7, so a warp writes 256 consecutive outputs (1 KiB fp32 or
// 512 B fp16) with 16-byte stores.  Each value is (d*sc)*q - dmin*m with every
// product and the difference rounded to nearest in fp32 (no contraction), the
// fp16 output is that fp32 value rounded to nearest even.
#include "common.cuh"
#include "internal.h"

namespace jllm {
namespace {

template <bool F16>
__global__ void __launch_bounds__(256) q4k_dequant_kernel(const uint8_t* __restrict__ W, void* __restrict__ out,
                                                          int64_t nblocks) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // lane l: weights i0 = 8l .. 8l+7; chunk c = i0/64, position r = i0%64.
  const int i0 = 8 * lane, c = i0 >> 6, r = i0 & 63;
  const int j = i0 >> 5;           // sub-block
  const bool high = r >= 32;       // high nibbles (sub-block 2c+1)
  const int byte0 = 32 * c + (r & 31);
  for (int64_t b = warp0; b < nblocks; b += nwarps) {
    const uint8_t* blk = W + b * BLOCK_BYTES;
    const uint4 hd = ldg_stream(blk);
    const uint2 qv = *reinterpret_cast<const uint2*>(blk + 16 + byte0);  // 8 code bytes
    uint32_t sc, m;
    q4k_scale_min(hd.y, hd.z, hd.w, j, sc, m);
    const float s = __fmul_rn(half_lo_to_float(hd.x), (float)sc);
    const float t = __fmul_rn(half_hi_to_float(hd.x), (float)m);
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t word = e < 4 ? qv.x : qv.y;
      const uint32_t byte = (word >> (8 * (e & 3))) & 0xffu;
      const uint32_t q = high ? (byte >> 4) : (byte & 15u);
      v[e] = q4k_value(s, t, q);
    }
    const int64_t o = b * QK + i0;
    if (F16) {
      uint4 pk;
      pk.x = (uint32_t)__half_as_ushort(__float2half_rn(v[0])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[1])) << 16);
      pk.y = (uint32_t)__half_as_ushort(__float2half_rn(v[2])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[3])) << 16);
      pk.z = (uint32_t)__half_as_ushort(__float2half_rn(v[4])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[5])) << 16);
      pk.w = (uint32_t)__half_as_ushort(__float2half_rn(v[6])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[7])) << 16);
      *reinterpret_cast<uint4*>(reinterpret_cast<__half*>(out) + o) = pk;
    } else {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

}  // namespace

cudaError_t launch_dequant(const void* w, void* out, bool f16, int64_t N, int64_t K, cudaStream_t s) {
  const DevInfo& dev = device_info();
  const int64_t nblocks = N * (K / QK);
  const int64_t want = (nblocks + 7) / 8;  // 8 warps per CTA
  const int64_t cap = (int64_t)dev.sm_count * 16;
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  if (f16)
    q4k_dequant_kernel<true><<<grid, 256, 0, s>>>((const uint8_t*)w, out, nblocks);
  else
    q4k_dequant_kernel<false><<<grid, 256, 0, s>>>((const uint8_t*)w, out, nblocks);
  return cudaGetLastError();
}

}  // namespace jllm

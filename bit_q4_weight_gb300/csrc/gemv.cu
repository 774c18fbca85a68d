// Q4_K dequant-fused GEMV (M = 1): y[n] = sum_k x[k] * w[n,k].
//
// The decode kernel of the genie-ai-runtime README ("At a glance", Kernels
// bullet: "INT4 dequant-fused GEMV"), re-designed for sm_103a:
//
//  * Work split.  A warp is four 8-lane groups; a group owns R weight rows.
//    Lane t of a group owns chunk c = t & 3 (64 weights: sub-blocks 2c and
//    2c+1) of every block kb with kb % 2 == t >> 2, so the 8 lanes cover two
//    144-byte blocks per step and walk the row two blocks at a time (split-K
//    over lanes).  Every lane issues 128-bit streaming loads of its block's
//    16-byte header and 32 code bytes straight from HBM; consecutive lanes read
//    consecutive bytes of the same two blocks.
//  * x is staged once per CTA in shared memory (16-byte units swizzled so the
//    eight lanes of a group read eight different bank groups) together with
//    the 32-element sums X_j of every sub-block.  A lane keeps its 64 x values
//    in registers for its R rows.
//  * Math.  Each code byte becomes two fp16 values 1024+q (low nibble) and
//    1024+16q (high nibble) with one LOP3 per pair; products with x are
//    accumulated in fp32 by the mixed-precision fma.rn.f32.f16 (exact
//    products).  Per sub-block j the offset is removed with the x sums:
//        sum_i w_i x_i = d*sc_j * (A_j - 1024*X_j) / (1 or 16) - dmin*m_j * X_j
//    which is the block value d*sc_j*q - dmin*m_j summed against x.
//  * Reduction.  Lane partials of a row are summed with three xor-shuffles
//    inside the group (deterministic order), lane 0 of the group stores y.
//  * Launch.  With programmatic dependent launch the first block's weights are
//    fetched before griddepcontrol.wait; x and y are touched only after it.
//
// SWIGLU mode computes the gate/up pair of a SwiGLU MLP in the same pass:
// weight row 2i of a group is gate row n, row 2i+1 is up row n, and the
// output is h[n] = silu(g) * u in fp16.
#include "common.cuh"
#include "internal.h"

namespace jllm {
namespace {

// acc += w0.lo*xa.lo + w1.lo*xa.hi + w0.hi*xb.lo + w1.hi*xb.hi  (fp16 x fp16 -> fp32)
__device__ __forceinline__ void fma4_h(float& acc, uint32_t w0, uint32_t w1, uint32_t xa, uint32_t xb) {
  asm("{\n .reg .b16 p0, p1, q0, q1, a0, a1, b0, b1;\n"
      " mov.b32 {p0, p1}, %1;\n mov.b32 {q0, q1}, %2;\n"
      " mov.b32 {a0, a1}, %3;\n mov.b32 {b0, b1}, %4;\n"
      " fma.rn.f32.f16 %0, p0, a0, %0;\n fma.rn.f32.f16 %0, q0, a1, %0;\n"
      " fma.rn.f32.f16 %0, p1, b0, %0;\n fma.rn.f32.f16 %0, q1, b1, %0;\n}"
      : "+f"(acc)
      : "r"(w0), "r"(w1), "r"(xa), "r"(xb));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(a), "r"(mask), "r"(orv));  // (a & b) | c
  return r;
}

// Position of 16-byte x unit (kb, c, b) in shared memory: the eight lanes
// of a group (kb parity p, chunk c) read unit b of their chunk in the same
// instruction; XOR-ing b with c | p<<2 puts them in eight bank groups.
__device__ __forceinline__ int x_unit_pos(int kb, int c, int b) {
  return (kb << 5) | (c << 3) | (b ^ (c | ((kb & 1) << 2)));
}

struct RowData {
  uint4 h, q0, q1;
};

__device__ __forceinline__ void load_row_block(RowData& d, const uint8_t* blk, int c) {
  d.h = ldg_stream(blk);
  d.q0 = ldg_stream(blk + 16 + 32 * c);
  d.q1 = ldg_stream(blk + 32 + 32 * c);
}

// Partial dot product of one lane's chunk (64 weights) of one block row.
__device__ __forceinline__ float chunk_dot(const RowData& d, const uint4 (&xv)[8], float Xlo, float Xhi,
                                           int c) {
  const uint32_t qw[8] = {d.q0.x, d.q0.y, d.q0.z, d.q0.w, d.q1.x, d.q1.y, d.q1.z, d.q1.w};
  float alo0 = 0.f, alo1 = 0.f, ahi0 = 0.f, ahi1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = qw[i];
    const uint32_t w8 = w >> 8;
    const uint32_t l02 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);   // 1024+q  (bytes 0,2 low)
    const uint32_t l13 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);  // 1024+q  (bytes 1,3 low)
    const uint32_t h02 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);   // 1024+16q (bytes 0,2 high)
    const uint32_t h13 = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);  // 1024+16q (bytes 1,3 high)
    const uint4 xl = xv[i >> 1];
    const uint4 xh = xv[4 + (i >> 1)];
    const uint32_t xla = (i & 1) ? xl.z : xl.x, xlb = (i & 1) ? xl.w : xl.y;
    const uint32_t xha = (i & 1) ? xh.z : xh.x, xhb = (i & 1) ? xh.w : xh.y;
    if (i & 1) {
      fma4_h(alo1, l02, l13, xla, xlb);
      fma4_h(ahi1, h02, h13, xha, xhb);
    } else {
      fma4_h(alo0, l02, l13, xla, xlb);
      fma4_h(ahi0, h02, h13, xha, xhb);
    }
  }
  const float alo = alo0 + alo1, ahi = ahi0 + ahi1;
  // scales and mins of sub-blocks 2c (lo) and 2c+1 (hi)
  const int hi = c >> 1, sh = 16 * (c & 1);
  const uint32_t A = d.h.y >> sh, B = d.h.z >> sh, E = d.h.w >> sh;
  const uint32_t sc_lo = hi ? ((E & 15u) | ((A >> 2) & 0x30u)) : (A & 63u);
  const uint32_t sc_hi = hi ? (((E >> 8) & 15u) | ((A >> 10) & 0x30u)) : ((A >> 8) & 63u);
  const uint32_t m_lo = hi ? (((E >> 4) & 15u) | ((B >> 2) & 0x30u)) : (B & 63u);
  const uint32_t m_hi = hi ? (((E >> 12) & 15u) | ((B >> 10) & 0x30u)) : ((B >> 8) & 63u);
  const float dd = half_lo_to_float(d.h.x), dm = half_hi_to_float(d.h.x);
  const float s_lo = dd * (float)sc_lo, s_hi = dd * (float)sc_hi * 0.0625f;
  const float t_lo = dm * (float)m_lo, t_hi = dm * (float)m_hi;
  float r = s_lo * fmaf(-1024.f, Xlo, alo);
  r = fmaf(-t_lo, Xlo, r);
  r = fmaf(s_hi, fmaf(-1024.f, Xhi, ahi), r);
  r = fmaf(-t_hi, Xhi, r);
  return r;
}

template <int R, int WPC, bool SWIGLU>
__global__ void __launch_bounds__(WPC * 32) q4k_gemv_kernel(const uint8_t* __restrict__ W0,
                                                            const uint8_t* __restrict__ W1,
                                                            const __half* __restrict__ x,
                                                            void* __restrict__ y, int N, int NB) {
  extern __shared__ uint4 gemv_smem[];
  uint4* xs = gemv_smem;                                          // NB*32 units
  float* Xs = reinterpret_cast<float*>(gemv_smem + (size_t)NB * 32);  // NB*8 sums

  constexpr int RP = SWIGLU ? R / 2 : R;  // output rows per group
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane >> 3, t = lane & 7, kp = t >> 2, c = t & 3;
  const int64_t nbase = ((int64_t)blockIdx.x * WPC + warp) * (4 * RP) + (int64_t)grp * RP;
  const int64_t row_bytes = (int64_t)NB * BLOCK_BYTES;

  const uint8_t* rowp[R];
  bool valid[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t n = SWIGLU ? nbase + r / 2 : nbase + r;
    const uint8_t* base = (SWIGLU && (r & 1)) ? W1 : W0;
    valid[r] = n < N;
    rowp[r] = base + (valid[r] ? n : 0) * row_bytes;
  }

  // Weights do not depend on the previous kernel: fetch the first block now.
  RowData cur[R];
  if (kp < NB) {
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (valid[r]) load_row_block(cur[r], rowp[r] + (int64_t)kp * BLOCK_BYTES, c);
  }

  pdl_wait();

  // Stage x (swizzled) and the sub-block sums X_j.
  const int nthreads = WPC * 32;
  for (int u = threadIdx.x; u < NB * 32; u += nthreads) {
    const int kb = u >> 5, cc = (u >> 3) & 3, b = u & 7;
    xs[x_unit_pos(kb, cc, b)] = ldg_nc(x + (size_t)u * 8);
  }
  for (int sb = threadIdx.x; sb < NB * 8; sb += nthreads) {
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 u4 = ldg_nc(x + (size_t)sb * 32 + v * 8);
      const uint32_t wv[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s += half_lo_to_float(wv[e]);
        s += half_hi_to_float(wv[e]);
      }
    }
    Xs[sb] = s;
  }
  __syncthreads();
  pdl_launch_dependents();

  float acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.f;

  for (int kb = kp; kb < NB; kb += 2) {
    RowData nxt[R];
    const bool more = kb + 2 < NB;
    if (more) {
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (valid[r]) load_row_block(nxt[r], rowp[r] + (int64_t)(kb + 2) * BLOCK_BYTES, c);
    }
    uint4 xv[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) xv[b] = xs[x_unit_pos(kb, c, b)];
    const float2 X = *reinterpret_cast<const float2*>(&Xs[kb * 8 + 2 * c]);
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (valid[r]) acc[r] += chunk_dot(cur[r], xv, X.x, X.y, c);
    if (more) {
#pragma unroll
      for (int r = 0; r < R; ++r) cur[r] = nxt[r];
    }
  }

#pragma unroll
  for (int r = 0; r < R; ++r) {
    float v = acc[r];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    acc[r] = v;
  }
  if (t == 0) {
    if (SWIGLU) {
#pragma unroll
      for (int i = 0; i < RP; ++i) {
        const int64_t n = nbase + i;
        if (n < N) {
          const float g = acc[2 * i], u = acc[2 * i + 1];
          const float h = g / (1.0f + expf(-g)) * u;
          reinterpret_cast<__half*>(y)[n] = __float2half_rn(h);
        }
      }
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (valid[r]) reinterpret_cast<float*>(y)[nbase + r] = acc[r];
    }
  }
}

template <int R, int WPC, bool SWIGLU>
cudaError_t launch_gemv_cfg(const void* w0, const void* w1, const void* x, void* y, int64_t N, int64_t K,
                            cudaStream_t stream, bool pdl) {
  const int NB = (int)(K / QK);
  constexpr int RP = SWIGLU ? R / 2 : R;
  const int64_t rows_per_cta = 4LL * RP * WPC;
  const int64_t grid = (N + rows_per_cta - 1) / rows_per_cta;
  const size_t smem = (size_t)NB * 32 * 16 + (size_t)NB * 8 * 4;
  auto kern = q4k_gemv_kernel<R, WPC, SWIGLU>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(WPC * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, (const uint8_t*)w0, (const uint8_t*)w1, (const __half*)x, y, (int)N,
                            NB);
}

}  // namespace

// Pick rows per group (R) and warps per CTA so that the grid covers the GPU
// at least twice where the shape allows, preferring more rows per lane (more
// reuse of the x registers).
cudaError_t launch_gemv(const void* w0, const void* w1, const void* x, void* y, int64_t N, int64_t K,
                        cudaStream_t stream) {
  const DevInfo& dev = device_info();
  const bool pdl = dev.pdl;
  const int64_t want = 2LL * dev.sm_count;
  if (w1 == nullptr) {
    if ((N + 63) / 64 >= want) return launch_gemv_cfg<4, 4, false>(w0, w1, x, y, N, K, stream, pdl);
    if ((N + 31) / 32 >= want) return launch_gemv_cfg<2, 4, false>(w0, w1, x, y, N, K, stream, pdl);
    if ((N + 15) / 16 >= want) return launch_gemv_cfg<2, 2, false>(w0, w1, x, y, N, K, stream, pdl);
    if ((N + 7) / 8 >= want) return launch_gemv_cfg<1, 2, false>(w0, w1, x, y, N, K, stream, pdl);
    return launch_gemv_cfg<1, 1, false>(w0, w1, x, y, N, K, stream, pdl);
  }
  if ((N + 31) / 32 >= want) return launch_gemv_cfg<4, 4, true>(w0, w1, x, y, N, K, stream, pdl);
  if ((N + 15) / 16 >= want) return launch_gemv_cfg<2, 4, true>(w0, w1, x, y, N, K, stream, pdl);
  if ((N + 7) / 8 >= want) return launch_gemv_cfg<2, 2, true>(w0, w1, x, y, N, K, stream, pdl);
  return launch_gemv_cfg<2, 1, true>(w0, w1, x, y, N, K, stream, pdl);
}

}  // namespace jllm

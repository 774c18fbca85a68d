// Q4_K dequant-fused GEMV (M = 1): y[n] = sum_k x[k] * w[n,k].
//
// The decode kernel of the genie-ai-runtime README ("At a glance", Kernels
// bullet: "INT4 dequant-fused GEMV"), re-designed for sm_103a:
//
//  * Streaming.  A CTA owns W*4*R weight rows.  Each warp's rows are one
//    contiguous byte range of W, copied HBM -> shared memory by a single
//    cp.async.bulk (TMA bulk copy) that completes on the warp's own mbarrier,
//    so the whole CTA's weights are in flight from the first cycle and every
//    warp starts as soon as its own rows land.  CTAs are kept small (tiles of
//    at most 48 KiB) so that several co-reside per SM and the next kernel in
//    the stream can start its copies while this one computes.
//  * Work split.  A warp is four 8-lane groups; a group owns R weight rows.
//    Lane t of a group owns chunk c = t & 3 (64 weights: sub-blocks 2c and
//    2c+1) of every block kb with kb % 2 == t >> 2, so the 8 lanes cover two
//    144-byte blocks per step with 128-bit shared-memory loads (conflict-free:
//    the eight lanes hit eight different bank groups) and walk the row two
//    blocks at a time (split-K over lanes).
//  * x arrives the same way (128-byte bulk copies into a padded layout whose
//    144-byte chunk stride puts the eight lanes of a group in eight different
//    bank groups); the 32-element sums X_j of every sub-block are formed from
//    shared memory.  A lane keeps its 64 x values in registers for its R rows.
//  * Math.  Each code byte becomes two fp16 values 1024+q (low nibble) and
//    1024+16q (high nibble) with one LOP3 per pair; products with x are
//    accumulated in fp32 by the mixed-precision fma.rn.f32.f16 (exact
//    products).  Per sub-block j the offset is removed with the x sums:
//        sum_i w_i x_i = d*sc_j * (A_j - 1024*X_j) / (1 or 16) - dmin*m_j * X_j
//    which is the block value d*sc_j*q - dmin*m_j summed against x.
//  * Reduction.  Lane partials of a row are summed with three xor-shuffles
//    inside the group (deterministic order), lane 0 of the group stores y.
//  * Launch.  With programmatic dependent launch the weight copies are issued
//    before griddepcontrol.wait; x and y are touched only after it.
//
// SWIGLU mode computes the gate/up pair of a SwiGLU MLP in the same pass:
// a group's weight rows alternate gate row n / up row n, and the output is
// h[n] = silu(g) * u in fp16.
#include <stdio.h>
#include <stdlib.h>

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

// Position (in 16-byte units) of unit b of the 128-byte x chunk (kb, c) in
// shared memory: chunks are stored 144 bytes apart, so the eight lanes of a
// group -- chunks 4*kb + c for kb = 2s, 2s+1 and c = 0..3, same b -- fall in
// eight different 16-byte bank groups (144 = 9 units, 9 = 1 mod 8).
__device__ __forceinline__ int x_unit_pos(int kb, int c, int b) { return (4 * kb + c) * 9 + b; }

struct RowData {
  uint4 h, q0, q1;
};

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

__device__ uint32_t g_gemv_error;
constexpr uint64_t GEMV_WAIT_LIMIT_NS = 2000000000ull;  // 2 s

// One CTA: W warps x 4 groups x R weight rows, K walked in chunks of KC
// blocks (one chunk whenever the rows fit, which covers the model shapes).
// Per chunk, warp w's rows arrive by bulk copy on the warp's own mbarrier --
// a single copy when the chunk is the whole row, since the warp's rows are
// then contiguous in W -- and each warp starts as soon as its rows land.
template <int R, int W, int KS, bool SWIGLU>
__global__ void __launch_bounds__(W * 32) q4k_gemv_kernel(const uint8_t* __restrict__ W0,
                                                          const uint8_t* __restrict__ W1,
                                                          const __half* __restrict__ x,
                                                          void* __restrict__ y, int N, int NB, int KC,
                                                          int trigger, int pre, int xbulk) {
  // KS = K-parts: the 4 groups of a warp form 4/KS row sets x KS K-parts; part
  // p of a row set takes block pairs p, p+KS, p+2KS, ...
  constexpr int RP = SWIGLU ? R / 2 : R;  // output rows per group
  constexpr int RS = 4 / KS;              // row sets per warp
  constexpr int ROWS_W = RS * R;          // weight rows per warp
  extern __shared__ __align__(128) uint8_t gemv_smem[];
  const int64_t row_bytes = (int64_t)NB * BLOCK_BYTES;   // global row pitch
  const int srow = KC * BLOCK_BYTES;                       // shared row pitch
  uint8_t* tile = gemv_smem;                                                  // W*ROWS_W rows x KC blocks
  uint4* xs = reinterpret_cast<uint4*>(tile + (size_t)W * ROWS_W * srow);   // KC*4 chunks of 9 units
  float* Xs = reinterpret_cast<float*>(xs + (size_t)KC * 36);               // KC*8 sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(Xs + (size_t)KC * 8);       // W weight barriers + 1 x barrier

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane >> 3, t = lane & 7, kp = t >> 2, c = t & 3;
  const int rset = grp / KS, kpart = grp % KS;
  const int64_t n_cta = (int64_t)blockIdx.x * (W * RS * RP);
  const int64_t n_warp = n_cta + (int64_t)warp * RS * RP;
  const int rows_w = (int)(N - n_warp < RS * RP ? (N - n_warp > 0 ? N - n_warp : 0) : RS * RP);
  const int nchunks = (NB + KC - 1) / KC;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w <= W; ++w) mbar_init(smem_u32(&bars[w]), 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  const uint32_t xbar = smem_u32(&bars[W]);
  // x chunk ch: 4*kc copies of 128 bytes into the padded layout, issued by warp 0.
  auto issue_x = [&](int ch) {
    const int kb0 = ch * KC, kc = NB - kb0 < KC ? NB - kb0 : KC;
    if (lane == 0) mbar_arrive_expect_tx(xbar, (uint32_t)kc * 512);
    __syncwarp();
    for (int i = lane; i < 4 * kc; i += 32)
      bulk_load(smem_u32(xs + (size_t)i * 9), x + ((size_t)kb0 * 4 + i) * 64, 128, xbar);
  };

  // Issue warp `warp`'s copies of chunk ch (lane 0 arms the barrier, lanes
  // 0..rows-1 copy one row each, or lane 0 copies the whole contiguous range).
  auto issue = [&](int ch) {
    if (rows_w == 0) return;
    const int kb0 = ch * KC, kc = NB - kb0 < KC ? NB - kb0 : KC;
    const uint32_t row_chunk = (uint32_t)kc * BLOCK_BYTES;
    const uint32_t bar = smem_u32(&bars[warp]);
    const uint32_t dst = smem_u32(tile + (size_t)warp * ROWS_W * srow);
    const uint32_t total = (uint32_t)rows_w * row_chunk * (SWIGLU ? 2 : 1);
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (kc == NB) {
      if (lane == 0) {
        bulk_load(dst, W0 + n_warp * row_bytes, (uint32_t)rows_w * row_chunk, bar);
        if (SWIGLU) bulk_load(dst + RS * RP * srow, W1 + n_warp * row_bytes, (uint32_t)rows_w * row_chunk, bar);
      }
    } else if (lane < rows_w) {
      const int64_t off = (n_warp + lane) * row_bytes + (int64_t)kb0 * BLOCK_BYTES;
      bulk_load(dst + lane * srow, W0 + off, row_chunk, bar);
      if (SWIGLU) bulk_load(dst + (RS * RP + lane) * srow, W1 + off, row_chunk, bar);
    }
  };

  // Weights do not depend on the previous kernel: start their copies now, and
  // let the next kernel in the stream launch and start its own.
  // Warps below `pre` fetch their rows before griddepcontrol.wait; the rest
  // after x, so that x does not queue behind the whole tile.
  if (warp < pre) issue(0);
  if (trigger == 1) pdl_launch_dependents();
  pdl_wait();
  if (warp >= pre) issue(0);
  if (xbulk && warp == 0) issue_x(0);
  float acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.f;
  const uint8_t* wtile = tile + (size_t)warp * ROWS_W * srow;
  const uint8_t* rowp[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = SWIGLU ? ((r & 1) ? RS * RP : 0) + rset * RP + r / 2 : rset * R + r;
    rowp[r] = wtile + (size_t)j * srow;
  }

  for (int ch = 0; ch < nchunks; ++ch) {
    const int kb0 = ch * KC, kc = NB - kb0 < KC ? NB - kb0 : KC;
    // Stage this chunk of x in the padded layout together with the sums X_j.
    // x normally comes through plain loads: the bulk-copy queue of the SM is
    // first-in first-out, and this CTA's (or the next kernel's) weight copies
    // would otherwise sit in front of it.
    if (xbulk) {
      if (!mbar_wait_bounded(xbar, ch & 1, nullptr, GEMV_WAIT_LIMIT_NS) && threadIdx.x == 0)
        atomicOr(&g_gemv_error, ERR_TIMEOUT);
    }
    for (int sb = threadIdx.x; sb < kc * 8; sb += W * 32) {
      const int kr = sb >> 3, j = sb & 7;
      float s = 0.f;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int pos = x_unit_pos(kr, j >> 1, 4 * (j & 1) + v);
        uint4 u4;
        if (xbulk) {
          u4 = xs[pos];
        } else {
          u4 = ldg_nc(x + (size_t)(kb0 + kr) * QK + 32 * j + 8 * v);
          xs[pos] = u4;
        }
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
    if (trigger == 2 && ch == 0) pdl_launch_dependents();

    if (rows_w > 0) {
      if (mbar_wait_bounded(smem_u32(&bars[warp]), ch & 1, nullptr, GEMV_WAIT_LIMIT_NS)) {
        for (int kr = 2 * kpart + kp; kr < kc; kr += 2 * KS) {
          uint4 xv[8];
#pragma unroll
          for (int b = 0; b < 8; ++b) xv[b] = xs[x_unit_pos(kr, c, b)];
          const float2 X = *reinterpret_cast<const float2*>(&Xs[kr * 8 + 2 * c]);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint8_t* blk = rowp[r] + kr * BLOCK_BYTES;
            RowData d;
            d.h = *reinterpret_cast<const uint4*>(blk);
            d.q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
            d.q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
            acc[r] += chunk_dot(d, xv, X.x, X.y, c);
          }
        }
      } else if (lane == 0) {
        atomicOr(&g_gemv_error, ERR_TIMEOUT);
      }
    }
    if (ch + 1 < nchunks) {
      __syncthreads();  // every warp is done with this chunk's x and weights
      issue(ch + 1);
      if (xbulk && warp == 0) issue_x(ch + 1);
    }
  }

  if (trigger == 3) pdl_launch_dependents();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float v = acc[r];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    if (KS >= 2) v += __shfl_xor_sync(0xffffffffu, v, 8);
    if (KS == 4) v += __shfl_xor_sync(0xffffffffu, v, 16);
    acc[r] = v;
  }
  if (t == 0 && kpart == 0) {
    const int64_t nb = n_warp + (int64_t)rset * RP;
#pragma unroll
    for (int i = 0; i < RP; ++i) {
      const int64_t n = nb + i;
      if (n >= N) break;
      if (SWIGLU) {
        const float g = acc[2 * i], u = acc[2 * i + 1];
        reinterpret_cast<__half*>(y)[n] = __float2half_rn(g / (1.0f + expf(-g)) * u);
      } else {
        reinterpret_cast<float*>(y)[n] = acc[i];
      }
    }
  }
}

// ------------------------------------------------------------------------
// Streaming kernel.  One CTA per SM; a producer lane keeps S shared-memory
// stages of RT consecutive weight rows in flight (one bulk copy per stage, two
// in SWIGLU mode; the first S are issued before griddepcontrol.wait).
//
// Consumer lanes are "slices": a team of WPR = ceil(NB/4) warps covers one
// row, lane slot l = 32*w + lane owning sub-block j = l % 8 of block
// kb = l / 8 (32 weights: the low nibbles of chunk j/2's 32 code bytes for
// even j, the high nibbles for odd j).  The lane keeps its 32 x values in
// registers as 30-bit fixed point, x*2^e split into a signed high and an
// unsigned low 16-bit limb (e per sub-block, from the sub-block's largest
// |x|; fp16 values within 2^19 of that maximum convert exactly), so
//     sum_i q_i x_i = 2^-e * (2^15 * sum q_i*hi_i + sum q_i*lo_i)
// is formed with dp2a (two 16x8-bit products per instruction, int32
// accumulation: exact).  Code bytes need one AND per four weights (high
// nibbles are used as 16q and scaled back by 1/16).  Per row and sub-block:
//     y += d*sc_j * (that sum) - dmin*m_j * X_j,   X_j = sum of the 32 x values.
// Partials are reduced with xor-shuffles inside a warp and in a fixed order
// through shared memory across the team's warps.
template <int C, int WPR, int R, bool SWIGLU>
__global__ void __launch_bounds__((C + 1) * 32) q4k_gemv_stream_kernel(
    const uint8_t* __restrict__ W0, const uint8_t* __restrict__ W1, const __half* __restrict__ x,
    void* __restrict__ y, int N, int NB, int S, int trigger) {
  constexpr int RP = SWIGLU ? R / 2 : R;   // output rows per team and stage
  constexpr int NT = C / WPR;              // teams
  constexpr int RT = NT * RP;              // output rows per stage
  extern __shared__ __align__(128) uint8_t gemv_smem[];
  const int row_bytes = NB * BLOCK_BYTES;
  const int stage_bytes = RT * row_bytes * (SWIGLU ? 2 : 1);
  uint8_t* stages = gemv_smem;                                                         // S stages
  float* red = reinterpret_cast<float*>(stages + (size_t)S * stage_bytes);           // [2][NT][R][WPR]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + 2 * NT * R * WPR + 2);           // full[S], empty[S]

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ntiles = (N + RT - 1) / RT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&bars[i]), 1);
      mbar_init(smem_u32(&bars[S + i]), C);
    }
    fence_mbarrier_init();
  }
  __syncthreads();

  auto produce = [&](int i) -> bool {
    const int tile = blockIdx.x + i * gridDim.x;
    const int slot = i % S;
    if (i >= S && !mbar_wait_bounded(smem_u32(&bars[S + slot]), ((i / S) & 1) ^ 1, nullptr, GEMV_WAIT_LIMIT_NS)) {
      atomicOr(&g_gemv_error, ERR_TIMEOUT);
      return false;
    }
    const int64_t n0 = (int64_t)tile * RT;
    const int rows = (int)(N - n0 < RT ? N - n0 : RT);
    const uint32_t bytes = (uint32_t)rows * row_bytes;
    const uint32_t bar = smem_u32(&bars[slot]);
    const uint32_t dst = smem_u32(stages + (size_t)slot * stage_bytes);
    mbar_arrive_expect_tx(bar, SWIGLU ? 2 * bytes : bytes);
    bulk_load(dst, W0 + n0 * row_bytes, bytes, bar);
    if (SWIGLU) bulk_load(dst + RT * row_bytes, W1 + n0 * row_bytes, bytes, bar);
    return true;
  };
  const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------- producer --
    if (lane == 0) {
      for (int i = 0; i < my_tiles && i < S; ++i) produce(i);
      pdl_wait();
      if (trigger == 2) pdl_launch_dependents();
      for (int i = S; i < my_tiles; ++i)
        if (!produce(i)) break;
    }
    return;
  }

  // --------------------------------------------------------------- consumers --
  const int cw = warp - 1, team = cw / WPR, wt = cw % WPR;
  const int sl = wt * 32 + lane;            // slice index within the row
  const bool active = sl < 8 * NB;
  const int kb = sl >> 3, j = sl & 7, c = j >> 1, hs = j & 1;
  pdl_wait();
  // x of this lane's sub-block -> two 16-bit limbs of x * 2^e, and X_j
  uint32_t xh[16], xl[16];
  float Xj = 0.f, coef = 0.f;
  if (active) {
    const __half* xp = x + (size_t)kb * QK + 32 * j;
    uint4 xv[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) xv[b] = ldg_nc(xp + 8 * b);
    float xf[32];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t wv[4] = {xv[b].x, xv[b].y, xv[b].z, xv[b].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xf[8 * b + 2 * e] = half_lo_to_float(wv[e]);
        xf[8 * b + 2 * e + 1] = half_hi_to_float(wv[e]);
      }
    }
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      mx = fmaxf(mx, fabsf(xf[i]));
      Xj += xf[i];
    }
    // e: largest power of two with max|x| * 2^e < 2^30
    int ex = 0;
    if (mx > 0.f) {
      frexpf(mx, &ex);  // mx = f * 2^ex, f in [0.5, 1)
      ex = 30 - ex;
    }
    coef = ldexpf(hs ? 0.0625f : 1.0f, -ex);  // undo 2^e (and the 16 of high nibbles)
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const int v0 = __float2int_rn(ldexpf(xf[2 * p], ex));
      const int v1 = __float2int_rn(ldexpf(xf[2 * p + 1], ex));
      xh[p] = ((uint32_t)(v0 >> 15) & 0xffffu) | ((uint32_t)(v1 >> 15) << 16);
      xl[p] = ((uint32_t)v0 & 0x7fffu) | (((uint32_t)v1 & 0x7fffu) << 16);
    }
  }
  const uint32_t qmask = hs ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
  // scale/min fields of sub-block j: bytes a = s[j&3], b = s[(j&3)+4], e = s[(j&3)+8]
  const int fsh = 8 * (j & 3);

  int i = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
    const int slot = i % S;
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars[slot]), (i / S) & 1, nullptr,
                                                              GEMV_WAIT_LIMIT_NS));
    if (!ok) {
      if (lane == 0) atomicOr(&g_gemv_error, ERR_TIMEOUT);
      break;
    }
    const uint8_t* st = stages + (size_t)slot * stage_bytes;
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      acc[r] = 0.f;
      if (active) {
        const int jr = SWIGLU ? ((r & 1) ? RT : 0) + team * RP + r / 2 : team * R + r;
        const uint8_t* blk = st + (size_t)jr * row_bytes + kb * BLOCK_BYTES;
        const uint4 hd = *reinterpret_cast<const uint4*>(blk);
        const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        int H0 = 0, H1 = 0, L0 = 0, L1 = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint32_t qb = qw[w] & qmask;
          if (w & 1) {
            asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(H1) : "r"(xh[2 * w]), "r"(qb));
            asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(H1) : "r"(xh[2 * w + 1]), "r"(qb));
            asm("dp2a.lo.u32.u32 %0, %1, %2, %0;" : "+r"(L1) : "r"(xl[2 * w]), "r"(qb));
            asm("dp2a.hi.u32.u32 %0, %1, %2, %0;" : "+r"(L1) : "r"(xl[2 * w + 1]), "r"(qb));
          } else {
            asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(H0) : "r"(xh[2 * w]), "r"(qb));
            asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(H0) : "r"(xh[2 * w + 1]), "r"(qb));
            asm("dp2a.lo.u32.u32 %0, %1, %2, %0;" : "+r"(L0) : "r"(xl[2 * w]), "r"(qb));
            asm("dp2a.hi.u32.u32 %0, %1, %2, %0;" : "+r"(L0) : "r"(xl[2 * w + 1]), "r"(qb));
          }
        }
        const float A = fmaf((float)(H0 + H1), 32768.f, (float)(L0 + L1));
        const uint32_t fa = (hd.y >> fsh) & 0xffu, fb = (hd.z >> fsh) & 0xffu, fe = (hd.w >> fsh) & 0xffu;
        const uint32_t sc = j < 4 ? (fa & 63u) : ((fe & 15u) | ((fa >> 6) << 4));
        const uint32_t mm = j < 4 ? (fb & 63u) : ((fe >> 4) | ((fb >> 6) << 4));
        const float dd = half_lo_to_float(hd.x), dm = half_hi_to_float(hd.x);
        acc[r] = fmaf(dd * (float)sc * coef, A, -(dm * (float)mm) * Xj);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));  // stage slot free for the producer
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float v = acc[r];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[r] = v;
    }
    if (WPR > 1) {
      float* rb = red + (size_t)((i & 1) * NT + team) * R * WPR;
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) rb[r * WPR + wt] = acc[r];
      }
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(WPR * 32) : "memory");
      if (wt == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float v = 0.f;
          for (int w = 0; w < WPR; ++w) v += rb[r * WPR + w];
          acc[r] = v;
        }
      }
    }
    if (wt == 0 && lane == 0) {
      const int64_t nb = (int64_t)tile * RT + team * RP;
#pragma unroll
      for (int ii = 0; ii < RP; ++ii) {
        const int64_t n = nb + ii;
        if (n >= N) break;
        if (SWIGLU) {
          const float gg = acc[2 * ii], u = acc[2 * ii + 1];
          reinterpret_cast<__half*>(y)[n] = __float2half_rn(gg / (1.0f + expf(-gg)) * u);
        } else {
          reinterpret_cast<float*>(y)[n] = acc[ii];
        }
      }
    }
  }
  if (trigger == 3) pdl_launch_dependents();
}

// Stages of a streaming CTA that fit `smem_cap` bytes (at most 8).
template <int C, int WPR, int R, bool SWIGLU>
int stream_stages(int NB, size_t smem_cap) {
  constexpr int RP = SWIGLU ? R / 2 : R;
  constexpr int RT = (C / WPR) * RP;
  const size_t stage = (size_t)RT * NB * BLOCK_BYTES * (SWIGLU ? 2 : 1);
  const size_t fixed = (size_t)(2 * (C / WPR) * R * WPR + 2) * 4 + 8 * 16 + 16;
  if (smem_cap <= fixed) return 0;
  const size_t n = (smem_cap - fixed) / stage;
  return (int)(n > 8 ? 8 : n);
}

template <int C, int WPR, int R, bool SWIGLU>
cudaError_t launch_gemv_stream(const void* w0, const void* w1, const void* x, void* y, int64_t N, int64_t K,
                               cudaStream_t stream, bool pdl, int trigger, int sms, size_t smem_cap) {
  const int NB = (int)(K / QK);
  constexpr int RP = SWIGLU ? R / 2 : R;
  constexpr int RT = (C / WPR) * RP;
  const int S = stream_stages<C, WPR, R, SWIGLU>(NB, smem_cap);
  if (S < 2 || 8 * NB > 32 * WPR) return cudaErrorInvalidValue;
  const size_t stage = (size_t)RT * NB * BLOCK_BYTES * (SWIGLU ? 2 : 1);
  const size_t smem = (size_t)S * stage + (size_t)(2 * (C / WPR) * R * WPR + 2) * 4 + 8 * 16 + 16;
  const int64_t ntiles = (N + RT - 1) / RT;
  const int grid = (int)(ntiles < sms ? ntiles : sms);
  auto kern = q4k_gemv_stream_kernel<C, WPR, R, SWIGLU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((C + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, (const uint8_t*)w0, (const uint8_t*)w1, (const __half*)x, y, (int)N,
                            NB, S, trigger);
}

// Tuning knobs read once from the environment:
//   JLLM_GEMV_CTAS_PER_SM  CTA target per SM for the configuration choice
//   JLLM_GEMV_CFG          "R,W,KS" forces one configuration (when built)
//   JLLM_GEMV_TRIGGER      where griddepcontrol.launch_dependents is issued:
//                          0 never, 1 at entry, 2 after x staging, 3 at the end
struct Knobs {
  int ctas_per_sm = 1;
  int R = 0, W = 0, KS = 0;
  int trigger = 1;
  int stream = 0;             // JLLM_GEMV_STREAM=1 selects the streaming kernel (off by default)
  int sC = 0, sR = 0, sKS = 0;  // JLLM_GEMV_SCFG="C,R" forces the consumer warps and rows of the streaming kernel
  int smem_kb = 100;          // JLLM_GEMV_SMEM_KB: shared-memory budget of a streaming CTA
  int pre_pct = 100;          // JLLM_GEMV_PRE: % of a CTA's warps whose rows are fetched before the wait
  int xbulk = 0;              // JLLM_GEMV_XBULK=1: x by bulk copies instead of plain loads
};
const Knobs& knobs() {
  static Knobs k = [] {
    Knobs v;
    if (const char* e = getenv("JLLM_GEMV_CTAS_PER_SM")) v.ctas_per_sm = atoi(e) < 1 ? 1 : atoi(e);
    if (const char* e = getenv("JLLM_GEMV_CFG")) sscanf(e, "%d,%d,%d", &v.R, &v.W, &v.KS);
    if (const char* e = getenv("JLLM_GEMV_TRIGGER")) v.trigger = atoi(e);
    if (const char* e = getenv("JLLM_GEMV_STREAM")) v.stream = atoi(e);
    if (const char* e = getenv("JLLM_GEMV_SCFG")) sscanf(e, "%d,%d", &v.sC, &v.sR);
    if (const char* e = getenv("JLLM_GEMV_SMEM_KB")) v.smem_kb = atoi(e);
    if (const char* e = getenv("JLLM_GEMV_PRE")) v.pre_pct = atoi(e);
    if (const char* e = getenv("JLLM_GEMV_XBULK")) v.xbulk = atoi(e);
    return v;
  }();
  return k;
}

// Blocks per K-chunk: the whole row when the warp tiles fit `tile_cap`.
template <int R, int W, int KS>
int gemv_kc(int NB, size_t tile_cap) {
  const size_t per_block = (size_t)W * (4 / KS) * R * BLOCK_BYTES;
  size_t kc = tile_cap / per_block;
  if (kc < 1) kc = 1;
  return (int)(kc < (size_t)NB ? kc : (size_t)NB);
}

template <int R, int W, int KS>
size_t gemv_smem_bytes(int KC) {
  return (size_t)W * (4 / KS) * R * KC * BLOCK_BYTES + (size_t)KC * 36 * 16 + (size_t)KC * 8 * 4 +
         (size_t)(W + 1) * 8;
}

constexpr size_t kGemvTileCap = 48 * 1024;

template <int R, int W, int KS, bool SWIGLU>
cudaError_t launch_gemv_cfg(const void* w0, const void* w1, const void* x, void* y, int64_t N, int64_t K,
                            cudaStream_t stream, bool pdl, int trigger, int pre_pct) {
  const int NB = (int)(K / QK);
  constexpr int RP = SWIGLU ? R / 2 : R;
  const int KC = gemv_kc<R, W, KS>(NB, kGemvTileCap);
  const int64_t rows_per_cta = (int64_t)(4 / KS) * RP * W;
  const int64_t grid = (N + rows_per_cta - 1) / rows_per_cta;
  const size_t smem = gemv_smem_bytes<R, W, KS>(KC);
  auto kern = q4k_gemv_kernel<R, W, KS, SWIGLU>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const int pre = (W * pre_pct + 99) / 100;
  return cudaLaunchKernelEx(&cfg, kern, (const uint8_t*)w0, (const uint8_t*)w1, (const __half*)x, y, (int)N,
                            NB, KC, trigger, pre, knobs().xbulk);
}

// The first configuration whose whole-row weight tile fits the tile cap and
// whose grid reaches the CTA target; else the last (smallest) one.
struct Cfg {
  int R, W, KS;
};

template <bool SWIGLU>
int pick(const Cfg* cfgs, int n, int64_t N, int NB, int sms, int ctas_per_sm) {
  for (int i = 0; i < n; ++i) {
    const int RP = SWIGLU ? cfgs[i].R / 2 : cfgs[i].R;
    const int64_t rows = (int64_t)(4 / cfgs[i].KS) * RP * cfgs[i].W;
    const size_t tile = (size_t)cfgs[i].W * (4 / cfgs[i].KS) * cfgs[i].R * NB * BLOCK_BYTES;
    if (tile <= kGemvTileCap && (N + rows - 1) / rows >= (int64_t)ctas_per_sm * sms) return i;
  }
  return n - 1;
}

#define JLLM_GEMV_CFGS(X)                                                                        \
  X(2, 8, 1) X(2, 4, 1) X(1, 8, 1) X(1, 4, 1) X(2, 8, 2) X(2, 4, 2) X(1, 8, 2) X(1, 4, 2)         \
      X(2, 8, 4) X(2, 4, 4) X(1, 8, 4) X(1, 4, 4) X(1, 2, 4) X(2, 2, 1) X(1, 2, 2) X(2, 2, 2)

}  // namespace

cudaError_t launch_gemv(const void* w0, const void* w1, const void* x, void* y, int64_t N, int64_t K,
                        cudaStream_t stream) {
  const DevInfo& dev = device_info();
  const bool pdl = dev.pdl;
  const int NB = (int)(K / QK);
  const Knobs& kn = knobs();
  const size_t scap = (size_t)kn.smem_kb * 1024;
  if (kn.stream && NB <= 40) {
    // Teams of WPR = ceil(NB/4) warps cover a row (one sub-block per lane);
    // C consumer warps (a multiple of WPR, at most 31); R rows per team.
    const int wpr = (NB + 3) / 4;
#define TRY(C_, WPR_, R_, SW_)                                                                                  \
  if (stream_stages<C_, WPR_, R_, SW_>(NB, scap) >= 2)                                                           \
    return launch_gemv_stream<C_, WPR_, R_, SW_>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, dev.sm_count, scap);
#define BY_WPR(R_, SW_)                                          \
  switch (wpr) {                                                 \
    case 1: { TRY(16, 1, R_, SW_) break; }                       \
    case 2: { TRY(16, 2, R_, SW_) break; }                       \
    case 3: { TRY(15, 3, R_, SW_) TRY(12, 3, R_, SW_) break; }   \
    case 4: { TRY(16, 4, R_, SW_) break; }                       \
    case 5: { TRY(15, 5, R_, SW_) TRY(10, 5, R_, SW_) break; }   \
    case 6: { TRY(18, 6, R_, SW_) TRY(12, 6, R_, SW_) break; }   \
    case 7: { TRY(14, 7, R_, SW_) break; }                       \
    case 8: { TRY(16, 8, R_, SW_) break; }                       \
    case 9: { TRY(18, 9, R_, SW_) break; }                       \
    case 10: { TRY(20, 10, R_, SW_) TRY(10, 10, R_, SW_) break; } \
    default: break;                                              \
  }
    if (w1 == nullptr) {
      if (kn.sR == 2) { BY_WPR(2, false) } else { BY_WPR(1, false) }
    } else {
      BY_WPR(2, true)
    }
#undef BY_WPR
#undef TRY
  }
  if (w1 == nullptr) {
    if (kn.R) {
#define X(R_, W_, KS_) \
  if (kn.R == R_ && kn.W == W_ && kn.KS == KS_) return launch_gemv_cfg<R_, W_, KS_, false>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
      JLLM_GEMV_CFGS(X)
#undef X
    }
    static const Cfg cfgs[] = {{2, 8, 1}, {2, 4, 1}, {1, 4, 1}, {1, 4, 2}, {1, 4, 4}, {1, 2, 4}};
    switch (pick<false>(cfgs, 6, N, NB, dev.sm_count, kn.ctas_per_sm)) {
      case 0: return launch_gemv_cfg<2, 8, 1, false>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
      case 1: return launch_gemv_cfg<2, 4, 1, false>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
      case 2: return launch_gemv_cfg<1, 4, 1, false>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
      case 3: return launch_gemv_cfg<1, 4, 2, false>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
      case 4: return launch_gemv_cfg<1, 4, 4, false>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
      default: return launch_gemv_cfg<1, 2, 4, false>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
    }
  }
  static const Cfg cfgs[] = {{4, 4, 1}, {2, 4, 1}, {2, 4, 2}, {2, 4, 4}};
  switch (pick<true>(cfgs, 4, N, NB, dev.sm_count, kn.ctas_per_sm)) {
    case 0: return launch_gemv_cfg<4, 4, 1, true>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
    case 1: return launch_gemv_cfg<2, 4, 1, true>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
    case 2: return launch_gemv_cfg<2, 4, 2, true>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
    default: return launch_gemv_cfg<2, 4, 4, true>(w0, w1, x, y, N, K, stream, pdl, kn.trigger, kn.pre_pct);
  }
}

cudaError_t read_clear_gemv_error(uint32_t* bits) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v));
  if (e == cudaSuccess && v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

}  // namespace jllm

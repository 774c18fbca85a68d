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
//  * Batches.  One launch may cover up to eight matrices that read the same
//    x (q/k/v of an attention block, gate/up of an MLP): each CTA finds its
//    matrix from the CTA ranges in the launch parameters.
//  * Work split.  A warp is four 8-lane groups; a group owns R weight rows.
//    Lane t of a group owns chunk c = t & 3 (64 weights: sub-blocks 2c and
//    2c+1) of every block kb with kb % 2 == t >> 2, so the 8 lanes cover two
//    144-byte blocks per step with 128-bit shared-memory loads (conflict-free:
//    the eight lanes hit eight different bank groups) and walk the row two
//    blocks at a time (split-K over lanes).
//  * x is loaded once per CTA with plain 128-bit loads, all issued before any
//    is used, into a padded shared layout whose 144-byte chunk stride puts
//    the eight lanes of a group in eight different bank groups; the
//    32-element sums X_j of every sub-block are formed on the way.
//  * Math.  Each code byte becomes two fp16 values by one AND per pair: the
//    low nibble left in place is the fp16 subnormal q*2^-24, the high nibble
//    left at bits 4..7 is 16q*2^-24.  Both are exact, with no offset to
//    remove afterwards.  Their products with x are accumulated in fp32 by the
//    mixed-precision fma.rn.f32.f16 (exact products), so per sub-block j
//        A_j = 2^-24 * sum_i q_i x_i        (or 16 * that for high nibbles)
//    and the staged x sums X_j are kept scaled by 2^-24 as well:
//        sum_i w_i x_i = 2^24 * ( d*sc_j * A_j (/16) - dmin*m_j * X_j*2^-24 )
//    which is the block value d*sc_j*q - dmin*m_j summed against x.  The
//    power-of-two scalings are exact; the row total is multiplied by 2^24
//    once at the end.  A code of 0 contributes an exact 0, so a sub-block
//    whose weights are all zero adds nothing, whatever its scale.  The
//    6-bit sc_j and m_j of a lane's two sub-blocks come out of the packed
//    bytes as one fp16 pair each (byte permute, masks, 1024 offset), and
//    d*sc_j, dmin*m_j are exact fp16 x fp16 products in fp32: no integer
//    conversions, and no lane-dependent branches.
//  * Reduction.  Lane partials of a row are summed with xor-shuffles inside
//    the group (deterministic order), lane 0 of the group stores y.
//  * Launch.  With programmatic dependent launch the weight copies are issued
//    before griddepcontrol.wait; x and y are touched only after it.
//
// SWIGLU mode computes the gate/up pair of a SwiGLU MLP in the same pass:
// a group's weight rows alternate gate row n / up row n, and the output is
// h[n] = silu(g) * u in fp16.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"
#include "q4k_dot.cuh"

namespace jllm {
namespace {

// acc += lo^2 + hi^2 of an fp16 pair (exact products, fp32 sums).
__device__ __forceinline__ void add_squares(float& acc, uint32_t h2) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %1;\n"
      " fma.rn.f32.f16 %0, a, a, %0;\n fma.rn.f32.f16 %0, b, b, %0;\n}"
      : "+f"(acc)
      : "r"(h2));
}

// fp16 pair (x * r * g) of an fp16 pair x, each product rounded in fp32 and
// the result once to fp16.
__device__ __forceinline__ uint32_t norm_pair(uint32_t h2, float r, float g0, float g1) {
  const float a = __fmul_rn(__fmul_rn(half_lo_to_float(h2), r), g0);
  const float b = __fmul_rn(__fmul_rn(half_hi_to_float(h2), r), g1);
  const __half2 o = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&o);
}


__device__ uint32_t g_gemv_error;
#ifndef JLLM_WAIT_LIMIT_NS
#define JLLM_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t GEMV_WAIT_LIMIT_NS = JLLM_WAIT_LIMIT_NS;  // 2 s (a test build shortens it)

#ifdef JLLM_FAULT_INJECTION
// Test builds only: when set, warp 0 of CTA 0 never issues its weight copy, so
// its bounded wait runs out and the GEMV's timeout path runs.
__device__ int g_fi_skip_w;
#endif

// The matrices of one launch.  Matrix i owns CTAs [cta0[i], cta0[i+1]).
struct GemvBatch {
  const uint8_t* w[kMaxGemvBatch];  // [n][NB] blocks
  void* y[kMaxGemvBatch];           // [n] fp32 (fp16 h in SWIGLU mode)
  int n[kMaxGemvBatch];
  int cta0[kMaxGemvBatch];
  int count;
  // Rotary epilogue (ROPE kernels): matrix i with bit i of rope_mask set holds
  // heads of 128 rows; hgamma[i] is its per-head RMSNorm weight [128]
  // (nullptr: no per-head norm).  Angle of pair j at position pos:
  // pos * rope_theta[j], rope_theta[j] = base^(-2j/128) formed on the host in fp64.
  const float* hgamma[kMaxGemvBatch];
  unsigned rope_mask;
  int rope_pos;
  float head_eps;
  double rope_theta[64];
};

constexpr int kHeadDim = 128;     // rows per head in the rotary epilogue
constexpr int kRopeCluster = 8;   // CTAs per head (16 rows = 8 rotation pairs each)

// One CTA: W warps x 4 groups x R weight rows, K walked in chunks of KC
// blocks (one chunk whenever the rows fit, which covers the model shapes).
// Per chunk, warp w's rows arrive by bulk copy on the warp's own mbarrier --
// a single copy when the chunk is the whole row, since the warp's rows are
// then contiguous in W -- and each warp starts as soon as its rows land.
template <int R, int W, int KS, bool SWIGLU, int MT, bool NORM, bool ROPE>
__global__ void __launch_bounds__(W * 32, 512 / (W * 32)) q4k_gemv_kernel(const __grid_constant__ GemvBatch batch,
                                                          const uint8_t* __restrict__ W1,
                                                          const __half* __restrict__ x, int NB, int KC,
                                                          int trigger, int pre, int M, int out_f16,
                                                          const float* __restrict__ gamma, float eps) {
  // MT = tokens per launch (M <= MT rows of x, row pitch K); a lane loads each of
  // its weight rows once per block and uses it for every token.
  // KS = K-parts: the 4 groups of a warp form 4/KS row sets x KS K-parts; part
  // p of a row set takes block pairs p, p+KS, p+2KS, ...
  constexpr int RP = SWIGLU ? R / 2 : R;  // output rows per group
  constexpr int RS = 4 / KS;              // row sets per warp
  constexpr int ROWS_W = RS * R;          // weight rows per warp
  constexpr int XU = 2;                   // x sub-blocks per thread whose loads are in flight together
  extern __shared__ __align__(128) uint8_t gemv_smem[];

  // This CTA's matrix (constant indices only: the parameters stay in the
  // parameter bank).
  const uint8_t* W0 = batch.w[0];
  void* y = batch.y[0];
  int N = batch.n[0], cta0 = 0;
  const float* hgamma = batch.hgamma[0];
  bool rope = ROPE && (batch.rope_mask & 1u);
#pragma unroll
  for (int i = 1; i < kMaxGemvBatch; ++i) {
    if (i < batch.count && (int)blockIdx.x >= batch.cta0[i]) {
      W0 = batch.w[i];
      y = batch.y[i];
      N = batch.n[i];
      cta0 = batch.cta0[i];
      if (ROPE) {
        hgamma = batch.hgamma[i];
        rope = (batch.rope_mask >> i) & 1u;
      }
    }
  }
  static_assert(!ROPE || (R == 1 && W == 4 && KS == 1 && !SWIGLU && MT == 1),
                "the rotary epilogue is laid out for 4 warps x 4 single-row groups");

  const int64_t row_bytes = (int64_t)NB * BLOCK_BYTES;   // global row pitch
  const int srow = KC * BLOCK_BYTES;                       // shared row pitch
  uint8_t* tile = gemv_smem;                                                  // W*ROWS_W rows x KC blocks
  uint4* xs = reinterpret_cast<uint4*>(tile + (size_t)W * ROWS_W * srow);   // MT x KC*4 chunks of 9 units
  float* Xs = reinterpret_cast<float*>(xs + (size_t)MT * KC * 36);          // MT x KC*8 sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(Xs + (size_t)MT * KC * 8);  // W weight barriers
  const int64_t K = (int64_t)NB * QK;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane >> 3, t = lane & 7, kp = t >> 2, c = t & 3;
  const int rset = grp / KS, kpart = grp % KS;
  const LaneDec L = lane_dec(c);
  const int64_t n_cta = (int64_t)((int)blockIdx.x - cta0) * (W * RS * RP);
  // Rotary matrices: the 8 CTAs of a cluster share one head; CTA rank cr owns
  // rows 8cr..8cr+7 (warps 0, 1) and their rotation partners 64+8cr..64+8cr+7
  // (warps 2, 3), four contiguous rows per warp.
  const int ccta = (int)blockIdx.x - cta0, crank = ccta & (kRopeCluster - 1);
  const int64_t n_warp = rope ? (int64_t)(ccta / kRopeCluster) * kHeadDim + (warp >= 2 ? kHeadDim / 2 : 0) +
                                    8 * crank + 4 * (warp & 1)
                              : n_cta + (int64_t)warp * RS * RP;
  const int rows_w = (int)(N - n_warp < RS * RP ? (N - n_warp > 0 ? N - n_warp : 0) : RS * RP);
  const int nchunks = (NB + KC - 1) / KC;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < W; ++w) mbar_init(smem_u32(&bars[w]), 1);
    fence_mbarrier_init();
  }
  __syncthreads();

  // Issue warp `warp`'s copies of chunk ch (lane 0 arms the barrier, lanes
  // 0..rows-1 copy one row each, or lane 0 copies the whole contiguous range).
  auto issue = [&](int ch) {
    if (rows_w == 0) return;
    const int kb0 = ch * KC, kc = NB - kb0 < KC ? NB - kb0 : KC;
    const uint32_t row_chunk = (uint32_t)kc * BLOCK_BYTES;
    const uint32_t bar = smem_u32(&bars[warp]);
    const uint32_t dst = smem_u32(tile + (size_t)warp * ROWS_W * srow);
    const uint32_t total = (uint32_t)rows_w * row_chunk * (SWIGLU ? 2 : 1);
    const uint64_t pol = l2_policy_evict_first();  // weights are read once per call
#ifdef JLLM_FAULT_INJECTION
    if (ch == 0 && warp == 0 && blockIdx.x == 0 && g_fi_skip_w) return;
#endif
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (kc == NB) {
      if (lane == 0) {
        bulk_load_hint(dst, W0 + n_warp * row_bytes, (uint32_t)rows_w * row_chunk, bar, pol);
        if (SWIGLU) bulk_load_hint(dst + RS * RP * srow, W1 + n_warp * row_bytes, (uint32_t)rows_w * row_chunk, bar, pol);
      }
    } else if (lane < rows_w) {
      const int64_t off = (n_warp + lane) * row_bytes + (int64_t)kb0 * BLOCK_BYTES;
      bulk_load_hint(dst + lane * srow, W0 + off, row_chunk, bar, pol);
      if (SWIGLU) bulk_load_hint(dst + (RS * RP + lane) * srow, W1 + off, row_chunk, bar, pol);
    }
  };

  // Weights do not depend on the previous kernel: start their copies now, and
  // let the next kernel in the stream launch and start its own.
  // Warps below `pre` fetch their rows before griddepcontrol.wait, the rest
  // after it.
  if (warp < pre) issue(0);
  if (trigger == 1) pdl_launch_dependents();
  // gamma is a weight too: pull its lines into L1 before the wait.
  const bool norm1 = NORM && nchunks == 1 && NB * 8 <= XU * W * 32;
  if (NORM)
    for (int sb = threadIdx.x; sb < NB * 8; sb += W * 32)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(gamma + (size_t)sb * 32));
  pdl_wait();
  if (warp >= pre) issue(0);
  float acc[R][MT];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
  const uint8_t* wtile = tile + (size_t)warp * ROWS_W * srow;
  const uint8_t* rowp[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = SWIGLU ? ((r & 1) ? RS * RP : 0) + rset * RP + r / 2 : rset * R + r;
    rowp[r] = wtile + (size_t)j * srow;
  }

  // RMSNorm prologue (one token): the CTA sums x^2 over all of K (exact fp16
  // squares, fp32 sums, a fixed reduction order) for r = 1/sqrt(mean + eps);
  // the staging below then stores fp16(x * r * gamma) and sums those.
  // When one pass of the staging loop covers all of x, the squares are summed
  // from the registers that pass loads instead (no second read of x).
  float rnorm = 1.f;
  __shared__ float red[W];
  if (NORM && !norm1) {
    float ss = 0.f;
    for (int sb = threadIdx.x; sb < NB * 8; sb += W * 32) {
      const __half* src = x + (size_t)sb * 32;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 u = ldg_nc(src + 8 * v);
        add_squares(ss, u.x);
        add_squares(ss, u.y);
        add_squares(ss, u.z);
        add_squares(ss, u.w);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) tot += red[w];
    rnorm = 1.f / sqrtf(tot / (float)K + eps);
  }

  for (int ch = 0; ch < nchunks; ++ch) {
    const int kb0 = ch * KC, kc = NB - kb0 < KC ? NB - kb0 : KC;
    // Stage this chunk of x (every token row) in the padded layout together with
    // the sums X_j: thread i takes sub-blocks i, i + W*32, ..., XU of them with
    // their loads in flight together.  Token rows m >= M read as zero.
    const int nsb = kc * 8;
    if (norm1) {
      // one token, normalised, one pass: load, reduce x^2 over the CTA, scale
      uint4 u[XU][4];
      float ss = 0.f;
#pragma unroll
      for (int q = 0; q < XU; ++q) {
        const int sb = threadIdx.x + q * W * 32;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          u[q][v] = sb < nsb ? ldg_nc(x + (size_t)sb * 32 + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
      }
      // gamma of the first sub-block, in flight together with x
      float4 g0[8];
#pragma unroll
      for (int v = 0; v < 8; ++v)
        g0[v] = (int)threadIdx.x < nsb ? __ldg(reinterpret_cast<const float4*>(gamma + (size_t)threadIdx.x * 32) + v)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < XU; ++q)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          add_squares(ss, u[q][v].x);
          add_squares(ss, u[q][v].y);
          add_squares(ss, u[q][v].z);
          add_squares(ss, u[q][v].w);
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) tot += red[w];
      rnorm = 1.f / sqrtf(tot / (float)K + eps);
#pragma unroll
      for (int q = 0; q < XU; ++q) {
        const int sb = threadIdx.x + q * W * 32;
        if (sb < nsb) {
          const float* g = gamma + (size_t)sb * 32;
          const int kr = sb >> 3, j = sb & 7;
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float4 ga = q == 0 ? g0[2 * v] : __ldg(reinterpret_cast<const float4*>(g + 8 * v));
            const float4 gb = q == 0 ? g0[2 * v + 1] : __ldg(reinterpret_cast<const float4*>(g + 8 * v + 4));
            uint4 t = u[q][v];
            t.x = norm_pair(t.x, rnorm, ga.x, ga.y);
            t.y = norm_pair(t.y, rnorm, ga.z, ga.w);
            t.z = norm_pair(t.z, rnorm, gb.x, gb.y);
            t.w = norm_pair(t.w, rnorm, gb.z, gb.w);
            xs[x_unit_pos(kr, j >> 1, 4 * (j & 1) + v)] = t;
            add_halves(s4[v], t.x);
            add_halves(s4[v], t.y);
            add_halves(s4[v], t.z);
            add_halves(s4[v], t.w);
          }
          Xs[sb] = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * kTwoM24;
        }
      }
    }
    for (int sb0 = threadIdx.x; !norm1 && sb0 < MT * nsb; sb0 += XU * W * 32) {
      uint4 u[XU][4];
#pragma unroll
      for (int q = 0; q < XU; ++q) {
        const int sb = sb0 + q * W * 32;
        const int m = MT == 1 ? 0 : sb / nsb, sl = MT == 1 ? sb : sb - m * nsb;
        if (sb < MT * nsb) {
          if (m < M) {
            const __half* src = x + (size_t)m * K + (size_t)(kb0 + (sl >> 3)) * QK + 32 * (sl & 7);
#pragma unroll
            for (int v = 0; v < 4; ++v) u[q][v] = ldg_nc(src + 8 * v);
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) u[q][v] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      if (NORM) {
#pragma unroll
        for (int q = 0; q < XU; ++q) {
          const int sb = sb0 + q * W * 32;
          if (sb < nsb) {
            const float* g = gamma + (size_t)(kb0 + (sb >> 3)) * QK + 32 * (sb & 7);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const float4 ga = __ldg(reinterpret_cast<const float4*>(g + 8 * v));
              const float4 gb = __ldg(reinterpret_cast<const float4*>(g + 8 * v + 4));
              u[q][v].x = norm_pair(u[q][v].x, rnorm, ga.x, ga.y);
              u[q][v].y = norm_pair(u[q][v].y, rnorm, ga.z, ga.w);
              u[q][v].z = norm_pair(u[q][v].z, rnorm, gb.x, gb.y);
              u[q][v].w = norm_pair(u[q][v].w, rnorm, gb.z, gb.w);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < XU; ++q) {
        const int sb = sb0 + q * W * 32;
        const int m = MT == 1 ? 0 : sb / nsb, sl = MT == 1 ? sb : sb - m * nsb;
        if (sb < MT * nsb) {
          const int kr = sl >> 3, j = sl & 7;
          // X_j in fp32: four chains of fp16 * 1 + fp32 (exact conversions)
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            xs[(size_t)m * KC * 36 + x_unit_pos(kr, j >> 1, 4 * (j & 1) + v)] = u[q][v];
            add_halves(s4[v], u[q][v].x);
            add_halves(s4[v], u[q][v].y);
            add_halves(s4[v], u[q][v].z);
            add_halves(s4[v], u[q][v].w);
          }
          Xs[(size_t)m * KC * 8 + sl] = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * kTwoM24;
        }
      }
    }
    __syncthreads();
    if (trigger == 2 && ch == 0) pdl_launch_dependents();

    if (rows_w > 0) {
      if (mbar_wait_bounded(smem_u32(&bars[warp]), ch & 1, nullptr, GEMV_WAIT_LIMIT_NS)) {
        for (int kr = 2 * kpart + kp; kr < kc; kr += 2 * KS) {
          RowData d[R];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint8_t* blk = rowp[r] + kr * BLOCK_BYTES;
            d[r].h = *reinterpret_cast<const uint4*>(blk);
            d[r].q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
            d[r].q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
          }
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4* xm = xs + (size_t)m * KC * 36;
            uint4 xv[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) xv[b] = xm[x_unit_pos(kr, c, b)];
            const float2 X = *reinterpret_cast<const float2*>(&Xs[(size_t)m * KC * 8 + kr * 8 + 2 * c]);
#pragma unroll
            for (int r = 0; r < R; ++r) chunk_dot(acc[r][m], d[r], xv, X.x, X.y, L);
          }
        }
      } else if (lane == 0) {
        atomicOr(&g_gemv_error, ERR_TIMEOUT);
      }
    }
    if (ch + 1 < nchunks) {
      __syncthreads();  // every warp is done with this chunk's x and weights
      issue(ch + 1);
    }
  }

  if (trigger == 3) pdl_launch_dependents();
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = acc[r][m];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      if (KS >= 2) v += __shfl_xor_sync(0xffffffffu, v, 8);
      if (KS == 4) v += __shfl_xor_sync(0xffffffffu, v, 16);
      acc[r][m] = v * kTwo24;  // the partials are in units of 2^-24 (exact rescaling)
    }
  }
  if (ROPE && rope) {
    // Rotary epilogue of one 16-row slice of a head: per-head RMSNorm (sum of
    // squares reduced over the cluster through distributed shared memory, in
    // rank order), then the rotation of pairs (j, j + 64), j = 8 cr + p.
    __shared__ float rv[16];
    __shared__ float hred[kRopeCluster];
    if (t == 0) rv[4 * warp + grp] = acc[0][0];
    __syncthreads();
    float r = 1.f;
    if (hgamma != nullptr) {
      if (threadIdx.x == 0) {
        float ss = 0.f;
#pragma unroll
        for (int l = 0; l < 16; ++l) ss = fmaf(rv[l], rv[l], ss);
        const uint32_t slot = smem_u32(&hred[crank]);
#pragma unroll
        for (int dst = 0; dst < kRopeCluster; ++dst) st_cluster_f32(mapa_shared(slot, (uint32_t)dst), ss);
      }
      cluster_sync_all();
      float tot = 0.f;
#pragma unroll
      for (int i = 0; i < kRopeCluster; ++i) tot += hred[i];
      r = 1.f / sqrtf(tot / (float)kHeadDim + batch.head_eps);
    }
    if (threadIdx.x < 8) {
      const int p = threadIdx.x, j = 8 * crank + p;
      float a = rv[p], b = rv[p + 8];
      if (hgamma != nullptr) {
        a = __fmul_rn(__fmul_rn(a, r), hgamma[j]);
        b = __fmul_rn(__fmul_rn(b, r), hgamma[j + kHeadDim / 2]);
      }
      // angle pos * theta_j and its reduction modulo 2 pi in fp64 (pi split in two parts, so
      // the remainder stays accurate at any 32-bit position), sine and cosine in fp32
      const double ang = (double)batch.rope_pos * batch.rope_theta[j];
      const double kq = rint(ang * 0.15915494309189535);           // 1 / (2 pi)
      double rr = fma(-kq, 6.283185307179586, ang);                  // 2 pi, high part
      rr = fma(-kq, 2.4492935982947064e-16, rr);                     // 2 pi, low part
      float sn, c;
      sincosf((float)rr, &sn, &c);
      float* yo = reinterpret_cast<float*>(y) + (int64_t)(ccta / kRopeCluster) * kHeadDim;
      yo[j] = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, sn));
      yo[j + kHeadDim / 2] = __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, sn));
    }
  } else if (t == 0 && kpart == 0) {
    const int64_t nb = n_warp + (int64_t)rset * RP;
#pragma unroll
    for (int i = 0; i < RP; ++i) {
      const int64_t n = nb + i;
      if (n >= N) break;
      if (SWIGLU) {
        const float g = acc[2 * i][0], u = acc[2 * i + 1][0];
        reinterpret_cast<__half*>(y)[n] = __float2half_rn(g / (1.0f + expf(-g)) * u);
      } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            if (out_f16) reinterpret_cast<__half*>(y)[(size_t)m * N + n] = __float2half_rn(acc[i][m]);
            else reinterpret_cast<float*>(y)[(size_t)m * N + n] = acc[i][m];
          }
        }
      }
    }
  }
}

// Launch-shape constants of the GEMV:
//   ctas_per_sm  CTA target per SM for the configuration choice
//   R, W, KS     one forced configuration (0: chosen per launch)
//   trigger      where griddepcontrol.launch_dependents is issued:
//                0 never, 1 at entry, 2 after x staging, 3 at the end
//   pre_pct      % of a CTA's warps whose rows are fetched before the wait
// They are fixed in the shipped library.  A build with -DJLLM_TUNING reads
// overrides once from the environment (JLLM_GEMV_CTAS_PER_SM, JLLM_GEMV_CFG
// = "R,W,KS", JLLM_GEMV_TRIGGER, JLLM_GEMV_PRE), for measurements only.
struct Knobs {
  int ctas_per_sm = 2;
  int R = 0, W = 0, KS = 0;
  int trigger = 1;
  int pre_pct = 100;
};
const Knobs& knobs() {
  static Knobs k = [] {
    Knobs v;
#ifdef JLLM_TUNING
    if (const char* e = getenv("JLLM_GEMV_CTAS_PER_SM")) v.ctas_per_sm = atoi(e) < 1 ? 1 : atoi(e);
    if (const char* e = getenv("JLLM_GEMV_CFG")) sscanf(e, "%d,%d,%d", &v.R, &v.W, &v.KS);
    if (const char* e = getenv("JLLM_GEMV_TRIGGER")) v.trigger = atoi(e);
    if (const char* e = getenv("JLLM_GEMV_PRE")) v.pre_pct = atoi(e);
#endif
    return v;
  }();
  return k;
}

// Shared bytes per block of K: the CTA's weight rows plus, per token, the x
// chunk (36 units of 16 bytes) and its 8 sub-block sums.
template <int R, int W, int KS, int MT>
constexpr size_t gemv_bytes_per_block() {
  return (size_t)W * (4 / KS) * R * BLOCK_BYTES + (size_t)MT * (36 * 16 + 8 * 4);
}

// Blocks per K-chunk: the whole row when it fits `cap`.
template <int R, int W, int KS, int MT>
int gemv_kc(int NB, size_t cap) {
  size_t kc = cap / gemv_bytes_per_block<R, W, KS, MT>();
  if (kc < 1) kc = 1;
  return (int)(kc < (size_t)NB ? kc : (size_t)NB);
}

template <int R, int W, int KS, int MT>
size_t gemv_smem_bytes(int KC) {
  return (size_t)KC * gemv_bytes_per_block<R, W, KS, MT>() + (size_t)W * 8;
}

constexpr size_t kGemvTileCap = 48 * 1024;      // weight tile of a one-token CTA
constexpr size_t kGemvMultiCap = 100 * 1024;    // weights + x of a multi-token CTA

// The matrices of a launch as the kernel sees them.
struct GemvJob {
  const void* const* w;
  void* const* y;
  const int64_t* n;
  int count;
  const void* w1;  // SwiGLU up matrix (count == 1), else nullptr
  const void* x;
  int64_t K;
  int M;           // tokens (rows of x), 1..kMaxGemvTokens
  int out_f16;
  const float* gamma = nullptr;  // RMSNorm weight [K] (one token only), else nullptr
  float eps = 0.f;
  // rotary epilogue (see GemvBatch)
  unsigned rope_mask = 0;
  const float* hgamma[kMaxGemvBatch] = {};
  int rope_pos = 0;
  double rope_base = 0.0;
  float head_eps = 0.f;
};

template <int R, int W, int KS, bool SWIGLU, int MT, bool NORM = false, bool ROPE = false>
cudaError_t launch_gemv_cfg(const GemvJob& job, cudaStream_t stream, bool pdl, int trigger, int pre_pct) {
  const int NB = (int)(job.K / QK);
  constexpr int RP = SWIGLU ? R / 2 : R;
  // One token: the weight tile alone is capped; several: weights and x together.
  const int KC = MT == 1 ? gemv_kc<R, W, KS, 0>(NB, kGemvTileCap) : gemv_kc<R, W, KS, MT>(NB, kGemvMultiCap);
  const int64_t rows_per_cta = (int64_t)(4 / KS) * RP * W;
  GemvBatch b = {};
  int64_t grid = 0;
  for (int i = 0; i < job.count; ++i) {
    b.w[i] = static_cast<const uint8_t*>(job.w[i]);
    b.y[i] = job.y[i];
    b.n[i] = (int)job.n[i];
    b.cta0[i] = (int)grid;
    grid += (job.n[i] + rows_per_cta - 1) / rows_per_cta;
  }
  b.count = job.count;
  if (ROPE) {
    for (int i = 0; i < job.count; ++i) {
      if (job.rope_mask >> i & 1u) {
        if (job.n[i] % kHeadDim) return cudaErrorInvalidValue;
        b.hgamma[i] = job.hgamma[i];
      }
      if (job.n[i] % (rows_per_cta * kRopeCluster)) return cudaErrorInvalidValue;  // whole clusters per matrix
    }
    b.rope_mask = job.rope_mask;
    b.rope_pos = job.rope_pos;
    b.head_eps = job.head_eps;
    for (int i = 0; i < kHeadDim / 2; ++i) b.rope_theta[i] = pow(job.rope_base, -2.0 * i / kHeadDim);
  }
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  const size_t smem = gemv_smem_bytes<R, W, KS, MT>(KC);
  static_assert(!NORM || (MT == 1 && !SWIGLU), "the RMSNorm prologue is one-token, single-output");
  auto kern = q4k_gemv_kernel<R, W, KS, SWIGLU, MT, NORM, ROPE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (ROPE) {  // the CTAs of one head form a cluster
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = kRopeCluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const int pre = (W * pre_pct + 99) / 100;
  return cudaLaunchKernelEx(&cfg, kern, b, static_cast<const uint8_t*>(job.w1), static_cast<const __half*>(job.x),
                            NB, KC, trigger, pre, job.M, job.out_f16, job.gamma, job.eps);
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

// Several tokens: one weight row per lane group (R = 1), the K split chosen
// like the one-token configurations.
template <int MT>
cudaError_t run_gemv_multi(const GemvJob& job, cudaStream_t stream, bool pdl, const Knobs& kn, int64_t rows, int NB,
                           int sms) {
  static const Cfg cfgs[] = {{1, 4, 1}, {1, 4, 2}, {1, 4, 4}, {1, 2, 4}};
  switch (pick<false>(cfgs, 4, rows, NB, sms, kn.ctas_per_sm)) {
    case 0: return launch_gemv_cfg<1, 4, 1, false, MT>(job, stream, pdl, kn.trigger, kn.pre_pct);
    case 1: return launch_gemv_cfg<1, 4, 2, false, MT>(job, stream, pdl, kn.trigger, kn.pre_pct);
    case 2: return launch_gemv_cfg<1, 4, 4, false, MT>(job, stream, pdl, kn.trigger, kn.pre_pct);
    default: return launch_gemv_cfg<1, 2, 4, false, MT>(job, stream, pdl, kn.trigger, kn.pre_pct);
  }
}

cudaError_t run_gemv(const GemvJob& job, cudaStream_t stream) {
  const DevInfo& dev = device_info();
  const bool pdl = dev.pdl;
  const int NB = (int)(job.K / QK);
  const Knobs& kn = knobs();
  int64_t rows = 0;
  for (int i = 0; i < job.count; ++i) rows += job.n[i];
  if (job.M > 1) {
    if (job.w1 != nullptr || job.count != 1 || job.gamma != nullptr) return cudaErrorInvalidValue;
    if (job.M <= 2) return run_gemv_multi<2>(job, stream, pdl, kn, rows, NB, dev.sm_count);
    if (job.M <= 4) return run_gemv_multi<4>(job, stream, pdl, kn, rows, NB, dev.sm_count);
    if (job.M <= 8) return run_gemv_multi<8>(job, stream, pdl, kn, rows, NB, dev.sm_count);
    return cudaErrorInvalidValue;
  }
  if (job.w1 == nullptr) {
    if (kn.R && job.gamma == nullptr) {
#define X(R_, W_, KS_) \
  if (kn.R == R_ && kn.W == W_ && kn.KS == KS_) return launch_gemv_cfg<R_, W_, KS_, false, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
      JLLM_GEMV_CFGS(X)
#undef X
    }
    static const Cfg cfgs[] = {{2, 8, 1}, {2, 4, 1}, {1, 4, 1}, {2, 4, 4}, {1, 4, 4}, {1, 2, 4}};
    if (job.gamma != nullptr) {  // RMSNorm prologue: its own instantiations
      switch (pick<false>(cfgs, 6, rows, NB, dev.sm_count, kn.ctas_per_sm)) {
        case 0: return launch_gemv_cfg<2, 8, 1, false, 1, true>(job, stream, pdl, kn.trigger, kn.pre_pct);
        case 1: return launch_gemv_cfg<2, 4, 1, false, 1, true>(job, stream, pdl, kn.trigger, kn.pre_pct);
        case 2: return launch_gemv_cfg<1, 4, 1, false, 1, true>(job, stream, pdl, kn.trigger, kn.pre_pct);
        case 3: return launch_gemv_cfg<2, 4, 4, false, 1, true>(job, stream, pdl, kn.trigger, kn.pre_pct);
        case 4: return launch_gemv_cfg<1, 4, 4, false, 1, true>(job, stream, pdl, kn.trigger, kn.pre_pct);
        default: return launch_gemv_cfg<1, 2, 4, false, 1, true>(job, stream, pdl, kn.trigger, kn.pre_pct);
      }
    }
    switch (pick<false>(cfgs, 6, rows, NB, dev.sm_count, kn.ctas_per_sm)) {
      case 0: return launch_gemv_cfg<2, 8, 1, false, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
      case 1: return launch_gemv_cfg<2, 4, 1, false, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
      case 2: return launch_gemv_cfg<1, 4, 1, false, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
      case 3: return launch_gemv_cfg<2, 4, 4, false, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
      case 4: return launch_gemv_cfg<1, 4, 4, false, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
      default: return launch_gemv_cfg<1, 2, 4, false, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
    }
  }
  static const Cfg cfgs[] = {{4, 4, 1}, {2, 4, 1}, {2, 4, 2}, {2, 4, 4}};
  switch (pick<true>(cfgs, 4, rows, NB, dev.sm_count, kn.ctas_per_sm)) {
    case 0: return launch_gemv_cfg<4, 4, 1, true, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
    case 1: return launch_gemv_cfg<2, 4, 1, true, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
    case 2: return launch_gemv_cfg<2, 4, 2, true, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
    default: return launch_gemv_cfg<2, 4, 4, true, 1>(job, stream, pdl, kn.trigger, kn.pre_pct);
  }
}

}  // namespace

cudaError_t launch_gemv(const void* w0, const void* w1, const void* x, void* y, int64_t N, int64_t K, int M,
                        bool y_f16, cudaStream_t stream) {
  const void* w[1] = {w0};
  void* yy[1] = {y};
  const int64_t n[1] = {N};
  return run_gemv(GemvJob{w, yy, n, 1, w1, x, K, M, y_f16 ? 1 : 0}, stream);
}

cudaError_t launch_gemv_batch(const void* const* w, void* const* y, const int64_t* N, int count, const void* x,
                              int64_t K, cudaStream_t stream) {
  if (count < 1 || count > kMaxGemvBatch) return cudaErrorInvalidValue;
  return run_gemv(GemvJob{w, y, N, count, nullptr, x, K, 1, 0}, stream);
}

cudaError_t launch_gemv_batch_rmsnorm(const void* const* w, void* const* y, const int64_t* N, int count,
                                      const void* x, const float* gamma, float eps, int64_t K, cudaStream_t stream) {
  if (count < 1 || count > kMaxGemvBatch || gamma == nullptr) return cudaErrorInvalidValue;
  GemvJob job{w, y, N, count, nullptr, x, K, 1, 0};
  job.gamma = gamma;
  job.eps = eps;
  return run_gemv(job, stream);
}

cudaError_t launch_gemv_qkv_rope(const void* const* w, void* const* y, const int64_t* N, int n_rope,
                                 const float* const* head_gamma, float head_eps, int pos, double rope_base,
                                 const void* x, const float* gamma, float eps, int64_t K, cudaStream_t stream) {
  if (n_rope < 1 || n_rope > 2) return cudaErrorInvalidValue;
  GemvJob job{w, y, N, 3, nullptr, x, K, 1, 0};
  job.gamma = gamma;
  job.eps = eps;
  job.rope_mask = (1u << n_rope) - 1u;
  for (int i = 0; i < n_rope; ++i) job.hgamma[i] = head_gamma[i];
  job.rope_pos = pos;
  job.rope_base = rope_base;
  job.head_eps = head_eps;
  const DevInfo& dev = device_info();
  const Knobs& kn = knobs();
  if (gamma != nullptr)
    return launch_gemv_cfg<1, 4, 1, false, 1, true, true>(job, stream, dev.pdl, kn.trigger, kn.pre_pct);
  return launch_gemv_cfg<1, 4, 1, false, 1, false, true>(job, stream, dev.pdl, kn.trigger, kn.pre_pct);
}

#ifdef JLLM_FAULT_INJECTION
cudaError_t fault_injection_set_gemv(int skip_w) { return cudaMemcpyToSymbol(g_fi_skip_w, &skip_w, sizeof(int)); }
#endif

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

// Q4_K dequant-fused GEMM for a few tokens (M <= 40): warp-level tensor
// cores (mma.sync m16n8k16, fp16 operands, fp32 accumulation) with the weights
// dequantised in registers.
//
// The short-prompt prefill of the genie-ai-runtime README ("At a glance",
// Kernels bullet: tensor-core prefill on Q4_K weights) sits on the HBM side of
// the balance point: each weight meets only M tokens, so the kernel must
// stream W at memory speed and do little per weight.  The tcgen05 GEMM pays a
// pipeline fill and one synchronisation round between its dequantising warps
// and its MMA thread per K step; with 5-20 steps per CTA at these M that is
// most of a launch.  Here every warp dequantises and multiplies its own rows,
// so the only hand-offs are the TMA stages.
//
//  * CTA: 128 weight rows x all tokens (T = 8 * NT >= M, one token tile) x a
//    K range.  Four consumer warps own 32 rows each (two 16-row MMA tiles that
//    share every x fragment); a fifth warp issues the TMA copies and forms the
//    per-sub-block sums of x.  Tiles with few rows split K over a thread-block
//    cluster whose CTAs add their partial sums in distributed shared memory
//    (fixed rank order: deterministic).  Two CTAs fit on an SM, so a launch's
//    weight copies start while the previous launch in the stream finishes
//    (programmatic dependent launch: W is issued before griddepcontrol.wait,
//    x after it).
//  * Stage (one 256-wide super-block column): raw W of 128 rows (3-D byte
//    view, 144-byte rows) and x as four 64-wide boxes of T tokens (128-byte
//    swizzle), both by TMA on one mbarrier.
//  * Weights as the A operand.  A 4-bit code masked in place is the fp16
//    subnormal q*2^-24 (low nibble) or 16q*2^-24 (high nibble); one fp16
//    multiply by 16*sc (low) or sc (high) gives exactly 16*sc*q*2^-24 (at most
//    15120 * 2^-24, exact in fp16).  So per super-block
//        sum_k w_k x_k = d * 2^20 * sum_k (16 sc q 2^-24) x_k  -  dmin * sum_j m_j X_j
//    with X_j the sum of x over sub-block j.  The first sum is one fp32
//    tensor-core accumulation per super-block, folded into the running total
//    with d * 2^20 (exact).  The second is one more MMA pair per super-block
//    accumulating straight into the total: dmin*m_j as an exact fp16 hi + lo
//    pair against -X_j as an fp16 hi + lo pair (X_j summed in fp32 by an MMA
//    against an indicator matrix).  Every product is exact; sums are fp32.
//  * K order inside an MMA: lane (g, t) of an m16n8k16 step holds code
//    positions 4t..4t+3 of its rows (one 32-bit word of codes per row gives
//    four steps: two positions each of two sub-blocks), and the x fragment
//    holds the same four positions of token g (one 64-bit shared load), so
//    the MMA's k order is a permutation of K applied to both operands.
//  * Domain: |dmin * m| <= 65504 and |sum of x over a sub-block of 32| <=
//    65504 (the fp16 hi parts), true of any model's weights and activations.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace jllm {
namespace {

__device__ uint32_t g_mma_error;
#ifndef JLLM_WAIT_LIMIT_NS
#define JLLM_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t MMA_WAIT_LIMIT_NS = JLLM_WAIT_LIMIT_NS;

#ifdef JLLM_FAULT_INJECTION
// Test builds only: when set, CTA 0 never issues its first x copies, so the
// waits on that stage run out and the timeout path runs.
__device__ int g_fi_skip_mma;
#endif

constexpr int MMA_ROWS = 128;                        // weight rows per CTA
constexpr int MMA_CWARPS = 4;                        // consumer warps, 32 rows each
constexpr int MMA_THREADS = (MMA_CWARPS + 1) * 32;   // + the copy / x-sum warp
constexpr int W_STAGE = MMA_ROWS * BLOCK_BYTES;      // 18432 bytes
constexpr int RED_PITCH = MMA_ROWS + 4;              // floats per token row of the partial sums
constexpr int kMmaMaxSplit = 16;                     // CTAs per cluster (above 8: non-portable)

template <int NT>
struct MmaCfg {
  static constexpr int T = 8 * NT;                   // tokens per CTA
  static constexpr int X_STAGE = 4 * T * 128;        // four 64-wide x boxes of T rows
  static constexpr int XS_STAGE = T * 32;            // per token: 8 sub-block sums as (hi, lo) fp16
  static constexpr int STAGE = X_STAGE + W_STAGE + XS_STAGE;
  // stages: as many as leave room for two CTAs per SM (at least 2, at most 4)
  static constexpr int S = 114000 / STAGE > 4 ? 4 : (114000 / STAGE < 2 ? 2 : 114000 / STAGE);
  static_assert(NT >= 1 && NT <= 5, "up to 40 tokens: two CTAs of 160 threads per SM need <= 168 registers");
  static constexpr int BAR_OFF = S * STAGE;
  static constexpr int SMEM = BAR_OFF + 3 * S * 8 + 1024;  // + barriers, + alignment slack
  static_assert(T * RED_PITCH * 4 <= S * X_STAGE, "partial sums must fit in the x stages");
  static_assert(X_STAGE % 1024 == 0, "swizzled x boxes need 1024-byte alignment");
};

// The matrices of one launch: matrix i owns row tiles [tile0[i], tile0[i+1]).
struct MmaParams {
  void* y[kMaxGemmBatch];
  int n[kMaxGemmBatch];
  int tile0[kMaxGemmBatch + 1];
  int count;
  int M;
  int NB;        // super-blocks per row (K / 256)
  int split;     // CTAs per tile (cluster size), each a K range
  int out_f16;
};
struct MmaWMaps {
  CUtensorMap w[kMaxGemmBatch];
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), b);
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Token (within a tile of 8) held by MMA column n.
__device__ __forceinline__ int tok_col(int n) { return ((n & 3) << 1) | (n >> 2); }

__device__ __forceinline__ void mma_fail(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_mma_error, 1u);
}

// fp16 pair (lo, hi) of the 6-bit fields bytes b0, b1 of word w: (1024 + f) as
// fp16 bits, minus 1024 (exact).
__device__ __forceinline__ __half2 six_bit_pair(uint32_t w, uint32_t sel) {
  const uint32_t h = __byte_perm(w, 0x64646464u, sel);
  return __hsub2(*reinterpret_cast<const __half2*>(&h), __float2half2_rn(1024.f));
}

// (16*sc_a, sc_b) of the 6-bit scales in bytes a, b of w: (1024 + sc) * (16, 1)
// - (16384, 1024), exact.
__device__ __forceinline__ __half2 scale_pair(uint32_t w, uint32_t sel) {
  const uint32_t h = __byte_perm(w, 0x64646464u, sel);
  return __hfma2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__float2half_rn(16.f), __float2half_rn(1.f)),
                 __halves2half2(__float2half_rn(-16384.f), __float2half_rn(-1024.f)));
}

template <int NT>
__global__ void __launch_bounds__(MMA_THREADS, 2)
    q4k_gemm_mma_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ MmaWMaps mw,
                        const __grid_constant__ MmaParams p) {
  using C = MmaCfg<NT>;
  constexpr int T = C::T, S = C::S;
  extern __shared__ uint8_t mma_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mma_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xst = smem;                       // S x-stages (1024-aligned boxes)
  uint8_t* wst = smem + S * C::X_STAGE;      // S W-stages
  uint8_t* xss = wst + S * W_STAGE;          // S x-sum stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int split = p.split;
  const int rank = (int)blockIdx.x % split;
  const int tile = (int)blockIdx.x / split;

  // This CTA's matrix (constant indices: the parameters stay in the parameter bank).
  const CUtensorMap* wmap = &mw.w[0];
  void* y = p.y[0];
  int N = p.n[0], t0 = p.tile0[0];
#pragma unroll
  for (int i = 1; i < kMaxGemmBatch; ++i)
    if (i < p.count && tile >= p.tile0[i]) {
      wmap = &mw.w[i];
      y = p.y[i];
      N = p.n[i];
      t0 = p.tile0[i];
    }
  const int n0 = (tile - t0) * MMA_ROWS;
  const int kb0 = rank * p.NB / split, kb1 = (rank + 1) * p.NB / split, nblk = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&bars[i]), 1);                    // full: W + x landed
      mbar_init(smem_u32(&bars[S + i]), MMA_CWARPS + 1);   // empty: every reader done
      mbar_init(smem_u32(&bars[2 * S + i]), 1);            // x sums written
    }
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  // MMA column n of a token tile holds token tok_col(n) of the tile: the lanes of
  // a half-warp (g = 0..3 or 4..7) then read x rows 0, 2, 4, 6 or 1, 3, 5, 7, whose
  // 128-byte swizzles spread their 64-bit loads over all 32 banks.
  const int pg = tok_col(g);
  // Swizzled byte offset, inside x row pg of a 64-wide box, of columns
  // 16q + 4t .. 16q + 4t + 3 (128-byte swizzle: 16-byte chunk ^ (row & 7)).
  uint32_t xoff[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) xoff[q] = ((uint32_t)((2 * q + (t >> 1)) ^ pg) << 4) | ((uint32_t)(t & 1) << 3);

  if (warp == MMA_CWARPS) {
    // ---- copies and x sums ----
    const bool leader = lane == 0;
    const int pre = nblk < S ? nblk : S;
    if (leader) {
      tma_prefetch_desc(&mx);
      tma_prefetch_desc(wmap);
      for (int i = 0; i < pre; ++i) {
        const uint32_t bar = smem_u32(&bars[i]);
        mbar_arrive_expect_tx(bar, (uint32_t)(W_STAGE + C::X_STAGE));
        tma_load_3d(smem_u32(wst + i * W_STAGE), wmap, bar, 0, kb0 + i, n0);
      }
    }
    pdl_wait();  // x is the previous kernel's output
    if (leader)
      for (int i = 0; i < pre; ++i) {
#ifdef JLLM_FAULT_INJECTION
        if (i == 0 && blockIdx.x == 0 && g_fi_skip_mma) continue;
#endif
        for (int h = 0; h < 4; ++h)
          tma_load_2d(smem_u32(xst + i * C::X_STAGE + h * T * 128), &mx, smem_u32(&bars[i]), (kb0 + i) * QK + 64 * h,
                      0);
      }
    int issued = pre, waited = 0;
    // indicator rows of the x-sum MMA: row j of A is all ones in the steps of sub-block j
    uint32_t ind[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ind[j] = g == j ? 0x3C003C00u : 0u;
    for (int i = 0; i < nblk; ++i) {
      const int slot = i % S;
      const uint32_t par = (uint32_t)(i / S) & 1u;
      if (!mbar_wait_warp(smem_u32(&bars[slot]), par, abort_v, MMA_WAIT_LIMIT_NS)) {
        if (leader) mma_fail(abort_v);
        break;
      }
      waited = i + 1;
      const uint8_t* xb = xst + slot * C::X_STAGE + pg * 128;
      uint8_t* xsb = xss + slot * C::XS_STAGE;  // rows by MMA column
      // NT independent accumulation chains, one per token tile
      float d[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = *reinterpret_cast<const uint2*>(xb + (j >> 1) * T * 128 + nt * 1024 + xoff[2 * (j & 1) + h2]);
            mma16816(d[nt], ind[j], 0u, ind[j], 0u, b.x, b.y);
          }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // d[nt][e] = sum of x over sub-block g of token nt*8 + 2t + e; stored negated as hi + lo
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = -d[nt][e];
          const __half hi = __float2half_rn(v);
          const __half lo = __float2half_rn(v - __half2float(hi));
          __half* row = reinterpret_cast<__half*>(xsb + (nt * 8 + 2 * t + e) * 32);
          row[(g >> 1) * 4 + (g & 1)] = hi;
          row[(g >> 1) * 4 + 2 + (g & 1)] = lo;
        }
      }
      __syncwarp();
      if (leader) {
        mbar_arrive(smem_u32(&bars[2 * S + slot]));
        mbar_arrive(smem_u32(&bars[S + slot]));
      }
      // Refill the previous block's slot once the consumers are done with it (the
      // sums of block i are ready before the consumers reach its end).
      const int r = i - 1;
      if (r >= 0 && r + S < nblk) {
        const int rslot = r % S;
        if (!mbar_wait_warp(smem_u32(&bars[S + rslot]), (uint32_t)(r / S) & 1u, abort_v, MMA_WAIT_LIMIT_NS)) {
          if (leader) mma_fail(abort_v);
          break;
        }
        if (leader) {
          const uint32_t bar = smem_u32(&bars[rslot]);
          const int kb = kb0 + r + S;
          mbar_arrive_expect_tx(bar, (uint32_t)(W_STAGE + C::X_STAGE));
          tma_load_3d(smem_u32(wst + rslot * W_STAGE), wmap, bar, 0, kb, n0);
          for (int h = 0; h < 4; ++h)
            tma_load_2d(smem_u32(xst + rslot * C::X_STAGE + h * T * 128), &mx, bar, kb * QK + 64 * h, 0);
        }
        issued = r + S + 1;
      }
    }
    // After a timeout: wait (bounded, whatever the abort flag) for copies still in flight.
    if (leader)
      for (int i = waited; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&bars[i % S]), (uint32_t)(i / S) & 1u, nullptr, MMA_WAIT_LIMIT_NS);
  } else {
    // ---- consumers: 32 rows each (rows g, g+8 | g+16, g+24 of the warp's 32) ----
    pdl_wait();
    float tot[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) tot[mt][nt][e] = 0.f;
    const int row0 = 32 * warp + g;
    for (int i = 0; i < nblk; ++i) {
      const int slot = i % S;
      const uint32_t par = (uint32_t)(i / S) & 1u;
      if (!mbar_wait_warp(smem_u32(&bars[slot]), par, abort_v, MMA_WAIT_LIMIT_NS)) {
        if (lane == 0) mma_fail(abort_v);
        break;
      }
      const uint8_t* wb = wst + slot * W_STAGE + row0 * BLOCK_BYTES;
      const uint8_t* xb = xst + slot * C::X_STAGE + pg * 128;
      // scales of the lane's four rows as (16 sc_2c, sc_2c+1) pairs (bytes 4..15 of
      // each block; d, dmin and the mins are read after the products)
      __half2 sp[4][4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const uint32_t s0 = *reinterpret_cast<const uint32_t*>(wb + rr * 8 * BLOCK_BYTES + 4);
        const uint32_t s2 = *reinterpret_cast<const uint32_t*>(wb + rr * 8 * BLOCK_BYTES + 12);
        const uint32_t sc_lo = s0 & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
        sp[rr][0] = scale_pair(sc_lo, 0x4140u);
        sp[rr][1] = scale_pair(sc_lo, 0x4342u);
        sp[rr][2] = scale_pair(sc_hi, 0x4140u);
        sp[rr][3] = scale_pair(sc_hi, 0x4342u);
      }
      float acc[2][NT][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int ph = 0; ph < 2; ++ph) {
          uint32_t pa[4], pb[4];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const uint32_t v = *reinterpret_cast<const uint32_t*>(wb + rr * 8 * BLOCK_BYTES + 16 + 32 * c + 16 * ph + 4 * t);
            pa[rr] = __byte_perm(v, 0u, 0x4140u);  // positions p, p+1 (low / high nibbles)
            pb[rr] = __byte_perm(v, 0u, 0x4342u);  // positions p+2, p+3
          }
#pragma unroll
          for (int hs = 0; hs < 2; ++hs) {
            const uint32_t mask = hs ? 0x00F000F0u : 0x000F000Fu;
            uint32_t a[4][2];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const __half2 s2 = hs ? __high2half2(sp[rr][c]) : __low2half2(sp[rr][c]);
              a[rr][0] = hmul2_u32(pa[rr] & mask, s2);
              a[rr][1] = hmul2_u32(pb[rr] & mask, s2);
            }
            const uint8_t* xc = xb + c * T * 128;
            const uint32_t xo = xoff[2 * hs + ph];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint2 b = *reinterpret_cast<const uint2*>(xc + nt * 1024 + xo);
              mma16816(acc[0][nt], a[0][0], a[1][0], a[0][1], a[1][1], b.x, b.y);
              mma16816(acc[1][nt], a[2][0], a[3][0], a[2][1], a[3][1], b.x, b.y);
            }
          }
        }
      // fold the super-block: total += d * 2^20 * acc
      float d20[4];
      uint32_t ah[4], al[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const uint4 h = *reinterpret_cast<const uint4*>(wb + rr * 8 * BLOCK_BYTES);
        d20[rr] = half_lo_to_float(h.x) * 1048576.f;
        // min term: dmin * m_j as an exact fp16 hi + lo pair (m_2t, m_2t+1 of this lane)
        const uint32_t mw = t < 2 ? (h.z & 0x3F3F3F3Fu) : (((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u));
        const __half2 m2 = six_bit_pair(mw, (t & 1) ? 0x4342u : 0x4140u);
        const __half2 dmin2 = __high2half2(*reinterpret_cast<const __half2*>(&h.x));
        const __half2 hi = __hmul2(m2, dmin2);
        const __half2 lo = __hfma2(m2, dmin2, __hneg2(hi));
        ah[rr] = *reinterpret_cast<const uint32_t*>(&hi);
        al[rr] = *reinterpret_cast<const uint32_t*>(&lo);
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          tot[mt][nt][0] = fmaf(d20[2 * mt], acc[mt][nt][0], tot[mt][nt][0]);
          tot[mt][nt][1] = fmaf(d20[2 * mt], acc[mt][nt][1], tot[mt][nt][1]);
          tot[mt][nt][2] = fmaf(d20[2 * mt + 1], acc[mt][nt][2], tot[mt][nt][2]);
          tot[mt][nt][3] = fmaf(d20[2 * mt + 1], acc[mt][nt][3], tot[mt][nt][3]);
        }
      // min term: dmin * m_j (hi + lo) against -X_j (hi + lo), into the total
      if (!mbar_wait_warp(smem_u32(&bars[2 * S + slot]), par, abort_v, MMA_WAIT_LIMIT_NS)) {
        if (lane == 0) mma_fail(abort_v);
        break;
      }
      const uint8_t* xsb = xss + slot * C::XS_STAGE + g * 32 + 8 * t;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint2 xs = *reinterpret_cast<const uint2*>(xsb + nt * 256);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma16816(tot[mt][nt], ah[2 * mt], ah[2 * mt + 1], al[2 * mt], al[2 * mt + 1], xs.x, xs.x);
          mma16816(tot[mt][nt], ah[2 * mt], ah[2 * mt + 1], al[2 * mt], al[2 * mt + 1], xs.y, xs.y);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[S + slot]));
    }
    // all consumers must be done with the x stages before they hold the partial sums
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(MMA_CWARPS * 32) : "memory");
    float* red = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = 32 * warp + 16 * mt + g;
        const int tk0 = nt * 8 + tok_col(2 * t), tk1 = nt * 8 + tok_col(2 * t + 1);
        red[tk0 * RED_PITCH + r] = tot[mt][nt][0];
        red[tk1 * RED_PITCH + r] = tot[mt][nt][1];
        red[tk0 * RED_PITCH + r + 8] = tot[mt][nt][2];
        red[tk1 * RED_PITCH + r + 8] = tot[mt][nt][3];
      }
  }
  // ---- partial sums -> y (the cluster's CTAs add theirs in rank order) ----
  __syncwarp();
  if (split > 1)
    cluster_sync_all();
  else
    __syncthreads();
  // This CTA's share: 4-row groups [ga, gb) of the 32, every token; the cluster's
  // partials are read with 16-byte loads, all in flight before they are added.
  const int ga = rank * (MMA_ROWS / 4) / split, gb = (rank + 1) * (MMA_ROWS / 4) / split, ng = gb - ga;
  const int M = p.M;
  uint32_t peer[kMmaMaxSplit];
  const uint32_t red_u32 = smem_u32(smem);
#pragma unroll
  for (int q = 0; q < kMmaMaxSplit; ++q)
    peer[q] = (split > 1 && q < split) ? mapa_shared(red_u32, (uint32_t)q) : red_u32;
  const bool vec = (N & 3) == 0;
  if (!*abort_v)
    for (int e = threadIdx.x; e < ng * M; e += MMA_THREADS) {
      const int tk = e / ng, r = 4 * (ga + e % ng);
      const int n = n0 + r;
      if (n >= N) continue;
      const uint32_t off = (uint32_t)(tk * RED_PITCH + r) * 4u;
      float4 v;
      if (split > 1) {
        float4 part[kMmaMaxSplit];
#pragma unroll
        for (int q = 0; q < kMmaMaxSplit; ++q)
          if (q < split) part[q] = ld_cluster_v4(peer[q] + off);
        v = part[0];
#pragma unroll
        for (int q = 1; q < kMmaMaxSplit; ++q)
          if (q < split) {
            v.x += part[q].x;
            v.y += part[q].y;
            v.z += part[q].z;
            v.w += part[q].w;
          }
      } else {
        v = *reinterpret_cast<const float4*>(smem + off);
      }
      const size_t o = (size_t)tk * N + n;
      if (vec && n + 3 < N) {
        if (p.out_f16) {
          const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
          uint2 u;
          u.x = *reinterpret_cast<const uint32_t*>(&a);
          u.y = *reinterpret_cast<const uint32_t*>(&b);
          *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(y) + o) = u;
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(y) + o) = v;
        }
      } else {
        const float vv[4] = {v.x, v.y, v.z, v.w};
        for (int i = 0; i < 4 && n + i < N; ++i) {
          if (p.out_f16)
            reinterpret_cast<__half*>(y)[o + i] = __float2half_rn(vv[i]);
          else
            reinterpret_cast<float*>(y)[o + i] = vv[i];
        }
      }
    }
  // no CTA leaves while its peers may still read its partial sums
  __syncwarp();
  if (split > 1) cluster_sync_all();
}

}  // namespace
}  // namespace jllm

// ---------------------------------------------------------------- host --
namespace jllm {
namespace {

// JLLM_GEMM_MMA_MAX_M (0..kGemmMmaMaxM, read once per process): when set, every M
// above the GEMV threshold and at most this value takes this kernel, whatever
// the shape.  -1: not set.
int forced_max_m() {
  static const int v = []() {
    const char* e = getenv("JLLM_GEMM_MMA_MAX_M");
    if (!e) return -1;
    const long x = strtol(e, nullptr, 10);
    return (x >= 0 && x <= kGemmMmaMaxM) ? (int)x : -1;
  }();
  return v;
}

// Clusters of `cs` CTAs of the NT-kernel that can be resident at once (cached per
// device, NT and cluster size; 0 when the query fails).
template <int NT>
int max_clusters(int cs) {
  struct Entry {
    int dev, cs, n;
  };
  static Entry cache[32];
  static int used = 0;
  static std::mutex mu;
  const int dev = device_info().device;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].cs == cs) return cache[i].n;
  auto kern = q4k_gemm_mma_kernel<NT>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MmaCfg<NT>::SMEM) == cudaSuccess &&
      (cs <= 8 || cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3(MMA_THREADS);
    cfg.dynamicSmemBytes = MmaCfg<NT>::SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)cs;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a refused query leaves no sticky error behind
  if (used < 32) cache[used++] = Entry{dev, cs, n};
  return n;
}

int max_clusters_for(int NT, int cs) {
  switch (NT) {
    case 1: return max_clusters<1>(cs);
    case 2: return max_clusters<2>(cs);
    case 3: return max_clusters<3>(cs);
    case 4: return max_clusters<4>(cs);
    default: return max_clusters<5>(cs);
  }
}

template <int NT>
cudaError_t launch_mma_nt(const CUtensorMap& mx, const MmaWMaps& mw, const MmaParams& p, int grid, cudaStream_t s) {
  auto kern = q4k_gemm_mma_kernel<NT>;
  constexpr int smem = MmaCfg<NT>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && p.split > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(MMA_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (p.split > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)p.split;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (device_info().pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, mx, mw, p);
}

}  // namespace

bool gemm_mma_takes(int64_t M, const int64_t* N, int count) {
  if (M < 1 || M > kGemmMmaMaxM) return false;
  const int forced = forced_max_m();
  if (forced >= 0) return M <= forced;
  // Measured against the tcgen05 GEMM on the layer shapes (2560 -> 6144, 4096 ->
  // 2560, 2560 -> 19456, 9728 -> 2560): faster on every shape up to 24 tokens;
  // at 25..40 tokens where the weights make at most 64 tiles of 128 rows (q/k/v,
  // o, down; not the 152 tiles of gate/up).
  if (M <= 24) return true;
  int64_t tiles = 0;
  for (int b = 0; b < count; ++b) tiles += (N[b] + MMA_ROWS - 1) / MMA_ROWS;
  return tiles <= 64;
}

cudaError_t launch_gemm_mma(const void* const* w, const int64_t* N, int count, const void* x, void* const* y,
                            bool y_f16, int64_t M, int64_t K, cudaStream_t s) {
  if (M < 1 || M > kGemmMmaMaxM || count < 1 || count > kMaxGemmBatch || K < QK || K % QK) return cudaErrorInvalidValue;
  const DevInfo& di = device_info();
  if (di.err != cudaSuccess) return di.err;
  const int NT = (int)((M + 7) / 8);
  CUtensorMap mx;
  MmaWMaps mw;
  MmaParams p = {};
  cudaError_t e = tma_map_x(x, M, K, 8 * NT, &mx);
  int tiles = 0;
  for (int b = 0; b < count && e == cudaSuccess; ++b) {
    e = tma_map_w(w[b], N[b], K, MMA_ROWS, &mw.w[b]);
    p.y[b] = y[b];
    p.n[b] = (int)N[b];
    p.tile0[b] = tiles;
    tiles += (int)((N[b] + MMA_ROWS - 1) / MMA_ROWS);
  }
  if (e != cudaSuccess) return e;
  for (int b = count; b <= kMaxGemmBatch; ++b) p.tile0[b] = tiles;
  p.count = count;
  p.M = (int)M;
  p.NB = (int)(K / QK);
  p.out_f16 = y_f16 ? 1 : 0;
  // Split K over a cluster so that the launch has about two CTAs per SM, lowered
  // until every cluster is resident at once (a second wave of clusters doubles a
  // launch), then the smallest split with the same largest share of super-blocks
  // per CTA (fewer CTAs and peers for the same critical path: 10 super-blocks
  // over 5 CTAs rather than 2, 2, 2, 2, 1, 1 over 6).
  int split = (2 * di.sm_count + tiles / 2) / tiles;
  if (split > kMmaMaxSplit) split = kMmaMaxSplit;
  if (split > p.NB) split = p.NB;
  if (split < 1) split = 1;
  while (split > 1 && max_clusters_for(NT, split) < tiles) --split;
  const int share = (p.NB + split - 1) / split;
  while (split > 1 && (p.NB + split - 2) / (split - 1) == share) --split;
  p.split = split;
  const int grid = tiles * split;
  switch (NT) {
    case 1: return launch_mma_nt<1>(mx, mw, p, grid, s);
    case 2: return launch_mma_nt<2>(mx, mw, p, grid, s);
    case 3: return launch_mma_nt<3>(mx, mw, p, grid, s);
    case 4: return launch_mma_nt<4>(mx, mw, p, grid, s);
    default: return launch_mma_nt<5>(mx, mw, p, grid, s);
  }
}

#ifdef JLLM_FAULT_INJECTION
cudaError_t fault_injection_set_mma(int skip) { return cudaMemcpyToSymbol(g_fi_skip_mma, &skip, sizeof(int)); }
#endif

cudaError_t read_clear_mma_error(uint32_t* bits) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_mma_error, sizeof(v));
  if (e == cudaSuccess && v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_mma_error, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

}  // namespace jllm

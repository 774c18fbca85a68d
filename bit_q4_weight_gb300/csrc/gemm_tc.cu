// Q4_K dequant-fused GEMM on the sm_103a tensor cores: Y = X * dequant(W)^T.
//
// The prefill kernel of the genie-ai-runtime README ("At a glance", Kernels
// bullet: "tensor-core MMQ Q4_K prefill"), re-designed around TMA, tcgen05
// and tensor memory.
//
// Orientation.  The MMA computes D[128 weight rows][BN tokens] += A * B^T with
// A = the dequantised fp16 weight tile (M = 128 rows of W, K-major) and B = a
// tile of X (N = BN tokens, K-major).  Putting W on the MMA's M side means a
// weight is dequantised once per CTA and reused for BN tokens.  D lives in
// tensor memory (lane = weight row, column = token, fp32).
//
// Roles (320 threads):
//   warp 0  TMA producer: per 64-wide K step one X tile {64 k x BN tokens},
//           128-byte swizzled; per 256-wide block one raw W tile
//           {144 bytes x 1 block x 128 rows} through a 3-D byte view of W.
//   warp 1  TMEM allocation and the MMA issuer (one thread): four
//           tcgen05.mma (K = 16 each) per K step, tcgen05.commit frees the
//           stages.
//   warps 2-9  dequantisers, two threads per weight row (low / high nibbles
//           of the row's 32 code bytes for this step): form the 32 values
//           (d*sc)*q - dmin*m exactly as the fp32 dequant does (sc*q exactly
//           in fp16x2, then one fp32 fma per value), round to fp16 and store
//           them in the 128-byte-swizzle K-major layout the MMA descriptor
//           expects.  They then run the epilogue: tcgen05.ld of their 32 TMEM
//           lanes, store Y (fp32 / fp16) or silu(g)*u (fp16).
// Every wait is bounded; a wait that runs out sets the device error word and
// the CTA winds down (pending copies and MMAs are awaited, TMEM is freed).
#include <cudaTypedefs.h>

#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace jllm {
namespace {

__device__ uint32_t g_gemm_error;

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(a), "r"(mask), "r"(orv));  // (a & b) | c
  return r;
}

// Two dequantised fp16 weights from two offset codes h (fp16x2):
// p = h*scv + offv = sc*q (exact), w = fma(d, p, nt) in fp32, packed to fp16x2.
__device__ __forceinline__ uint32_t dq_pair(uint32_t h2, uint32_t scv, uint32_t offv, unsigned short d,
                                            float nt) {
  uint32_t p, out;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(p) : "r"(h2), "r"(scv), "r"(offv));
  asm("{\n .reg .b16 pl, ph;\n .reg .f32 a, b;\n mov.b32 {pl, ph}, %1;\n"
      " fma.rn.f32.f16 a, %2, pl, %3;\n fma.rn.f32.f16 b, %2, ph, %3;\n"
      " cvt.rn.f16x2.f32 %0, b, a;\n}"
      : "=r"(out)
      : "r"(p), "h"(d), "f"(nt));
  return out;
}

constexpr int TILE_N = 128;           // weight rows per CTA (MMA M)
constexpr int KSTEP = 64;             // K per stage (128 bytes of fp16)
constexpr int A_STAGE_BYTES = TILE_N * KSTEP * 2;        // 16 KiB
constexpr int W_STAGE_BYTES = TILE_N * BLOCK_BYTES;      // 18 KiB
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s

struct GemmParams {
  void* y;
  int M, N, NB;
  int BN;          // tokens per CTA (MMA N), multiple of 16, <= 256
  int SX, SA, SW;  // stage counts of the X, A and raw-W rings
  uint32_t off_x, off_a, off_w, off_bar;  // shared-memory carve-up (bytes)
  uint32_t tmem_cols;
  int out_f16;
};

template <bool SWIGLU>
__global__ void __launch_bounds__(320, 1)
    q4k_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                       const __grid_constant__ CUtensorMap tmW1, const GemmParams p) {
  constexpr int NMAT = SWIGLU ? 2 : 1;
  extern __shared__ uint8_t gemm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sx = sbase + p.off_x, sa = sbase + p.off_a, sw = sbase + p.off_w;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  // barrier layout: x_full[SX] x_empty[SX] w_full[SW] w_empty[SW] a_full[SA] a_empty[SA] acc_full
  const uint32_t b_xfull = smem_u32(bars), b_xempty = b_xfull + 8 * p.SX;
  const uint32_t b_wfull = b_xempty + 8 * p.SX, b_wempty = b_wfull + 8 * p.SW;
  const uint32_t b_afull = b_wempty + 8 * p.SW, b_aempty = b_afull + 8 * p.SA;
  const uint32_t b_acc = b_aempty + 8 * p.SA;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * (p.SX + p.SW + p.SA) + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * TILE_N, m0 = blockIdx.y * p.BN;
  const int KS = p.NB * (256 / KSTEP);
  const uint32_t x_stage_bytes = (uint32_t)p.BN * KSTEP * 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.SX; ++i) {
      mbar_init(b_xfull + 8 * i, 1);
      mbar_init(b_xempty + 8 * i, 1);
    }
    for (int i = 0; i < p.SW; ++i) {
      mbar_init(b_wfull + 8 * i, 1);
      mbar_init(b_wempty + 8 * i, 8);
    }
    for (int i = 0; i < p.SA; ++i) {
      mbar_init(b_afull + 8 * i, 8);
      mbar_init(b_aempty + 8 * i, 1);
    }
    mbar_init(b_acc, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(&g_gemm_error, ERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer --
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmW0);
      if (SWIGLU) tma_prefetch_desc(&tmW1);
      int issued_x = 0, issued_w = 0;
      for (int ks = 0; ks < KS; ++ks) {
        if ((ks & 3) == 0) {
          const int kb = ks >> 2, s = kb % p.SW;
          if (!mbar_wait_bounded(b_wempty + 8 * s, ((kb / p.SW) & 1) ^ 1, abort_flag, WAIT_LIMIT_NS)) {
            fail();
            break;
          }
          mbar_arrive_expect_tx(b_wfull + 8 * s, W_STAGE_BYTES * NMAT);
          tma_load_3d(sw + (uint32_t)(s * NMAT) * W_STAGE_BYTES, &tmW0, b_wfull + 8 * s, 0, kb, n0);
          if (SWIGLU)
            tma_load_3d(sw + (uint32_t)(s * NMAT + 1) * W_STAGE_BYTES, &tmW1, b_wfull + 8 * s, 0, kb, n0);
          issued_w = kb + 1;
        }
        const int s = ks % p.SX;
        if (!mbar_wait_bounded(b_xempty + 8 * s, ((ks / p.SX) & 1) ^ 1, abort_flag, WAIT_LIMIT_NS)) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(b_xfull + 8 * s, x_stage_bytes);
        tma_load_2d(sx + (uint32_t)s * x_stage_bytes, &tmX, b_xfull + 8 * s, ks * KSTEP, m0);
        issued_x = ks + 1;
      }
      // Every copy this thread issued must have landed before the CTA exits.
      for (int i = issued_x - p.SX; i < issued_x; ++i)
        if (i >= 0) mbar_wait_bounded(b_xfull + 8 * (i % p.SX), (i / p.SX) & 1, nullptr, WAIT_LIMIT_NS);
      for (int i = issued_w - p.SW; i < issued_w; ++i)
        if (i >= 0) mbar_wait_bounded(b_wfull + 8 * (i % p.SW), (i / p.SW) & 1, nullptr, WAIT_LIMIT_NS);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer --
      const uint32_t idesc = umma_idesc_f16(TILE_N, p.BN);
      for (int ks = 0; ks < KS; ++ks) {
        const int s_a = ks % p.SA, s_x = ks % p.SX;
        if (!mbar_wait_bounded(b_afull + 8 * s_a, (ks / p.SA) & 1, abort_flag, WAIT_LIMIT_NS) ||
            !mbar_wait_bounded(b_xfull + 8 * s_x, (ks / p.SX) & 1, abort_flag, WAIT_LIMIT_NS)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sa + (uint32_t)(s_a * NMAT) * A_STAGE_BYTES;
        const uint32_t b0 = sx + (uint32_t)s_x * x_stage_bytes;
#pragma unroll
        for (int kk = 0; kk < KSTEP / 16; ++kk) {
          const uint64_t bd = umma_desc_sw128(b0 + 32 * kk);
          const uint32_t acc = (ks | kk) != 0;
          umma_f16(tmem, umma_desc_sw128(a0 + 32 * kk), bd, idesc, acc);
          if (SWIGLU) umma_f16(tmem + (p.tmem_cols >> 1), umma_desc_sw128(a0 + A_STAGE_BYTES + 32 * kk), bd, idesc, acc);
        }
        umma_commit(b_aempty + 8 * s_a);
        umma_commit(b_xempty + 8 * s_x);
      }
      umma_commit(b_acc);  // also tracks every MMA issued before an abort
      mbar_wait_bounded(b_acc, 0, nullptr, WAIT_LIMIT_NS);
    }
  } else {
    // ------------------------------------------------- dequant + epilogue --
    // Warps 2..9: warp w handles TMEM lane quarter q = w & 3 (rows 32q..32q+31)
    // and nibble side hs = (w - 2) >> 2: hs = 0 makes sub-block 2c (low
    // nibbles, k 0..31 of the step), hs = 1 sub-block 2c+1 (high nibbles,
    // k 32..63).
    const int q = warp & 3;
    const int hs = (warp - 2) >> 2;
    const int r = 32 * q + lane;  // weight row within the tile
    bool ok = true;
    for (int ks = 0; ks < KS && ok; ++ks) {
      const int kb = ks >> 2, c = ks & 3, s_w = kb % p.SW, s_a = ks % p.SA;
      // Waits are made warp-uniform so that a timeout leaves the warp converged.
      if (c == 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_wfull + 8 * s_w, (kb / p.SW) & 1, abort_flag, WAIT_LIMIT_NS));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_aempty + 8 * s_a, ((ks / p.SA) & 1) ^ 1, abort_flag, WAIT_LIMIT_NS));
      if (!ok) break;
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        const uint8_t* raw = smem + p.off_w + (size_t)(s_w * NMAT + mat) * W_STAGE_BYTES + (size_t)r * BLOCK_BYTES;
        const uint4 hd = *reinterpret_cast<const uint4*>(raw);
        const uint4 q0 = *reinterpret_cast<const uint4*>(raw + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(raw + 32 + 32 * c);
        uint32_t sc, m;
        q4k_scale_min(hd.y, hd.z, hd.w, 2 * c + hs, sc, m);
        // p = sc*q exactly in fp16 from the offset code h (1024+q or 1024+16q):
        //   p = h*sc - 1024*sc  or  p = h*(sc/16) - 64*sc   (one rounding of an
        //   exact integer <= 945).  Then w = fma(d, p, -dmin*m) in fp32 is the
        //   exact value rounded once, i.e. the fp32 dequant, rounded to fp16.
        const __half sch = __uint2half_rn(sc);
        const __half2 scv = __half2half2(hs ? __hmul(sch, __float2half(0.0625f)) : sch);
        const __half2 offv = __half2half2(__hmul(sch, __float2half(hs ? -64.f : -1024.f)));
        const uint32_t scv_u = *reinterpret_cast<const uint32_t*>(&scv);
        const uint32_t offv_u = *reinterpret_cast<const uint32_t*>(&offv);
        const unsigned short d16 = (unsigned short)(hd.x & 0xffffu);
        const float nt = -__fmul_rn(half_hi_to_float(hd.x), (float)m);
        const uint32_t mask = hs ? 0x00F000F0u : 0x000F000Fu;
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint8_t* arow = smem + p.off_a + (size_t)(s_a * NMAT + mat) * A_STAGE_BYTES + (size_t)r * 128;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          // output chunk j8 = 4*hs + jj holds k = 8*j8..8*j8+7: code bytes 8*jj..8*jj+7
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t w = qw[2 * jj + e];
            uint32_t wp;
            asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(wp) : "r"(w));  // bytes b0 b2 b1 b3
            pk[2 * e] = dq_pair(lop3_and_or(wp, mask, 0x64006400u), scv_u, offv_u, d16, nt);       // k, k+1
            pk[2 * e + 1] = dq_pair(lop3_and_or(wp >> 8, mask, 0x64006400u), scv_u, offv_u, d16, nt);  // k+2, k+3
          }
          const int j8 = 4 * hs + jj;
          *reinterpret_cast<uint4*>(arow + ((j8 ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(b_afull + 8 * s_a);
        if (c == 3) mbar_arrive(b_wempty + 8 * s_w);
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_acc, 0, abort_flag, WAIT_LIMIT_NS));
    if (!ok) {
      if (lane == 0) fail();
    } else {
      tc_fence_after();
      const int n = n0 + r;
      const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
      // the two warps of a lane quarter split the token columns in 32-wide chunks
      for (int cc = 32 * hs; cc < p.BN; cc += 64) {
        uint32_t v[32];
        tmem_ld32(lane_addr + cc, v);
        if (SWIGLU) {
          uint32_t u[32];
          tmem_ld32(lane_addr + (p.tmem_cols >> 1) + cc, u);
          if (n < p.N) {
            __half* y = reinterpret_cast<__half*>(p.y);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + cc + j;
              if (m < p.M && cc + j < p.BN) {
                const float g = __uint_as_float(v[j]), uu = __uint_as_float(u[j]);
                y[(size_t)m * p.N + n] = __float2half_rn(g / (1.0f + expf(-g)) * uu);
              }
            }
          }
        } else if (n < p.N) {
          if (p.out_f16) {
            __half* y = reinterpret_cast<__half*>(p.y);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + cc + j;
              if (m < p.M && cc + j < p.BN) y[(size_t)m * p.N + n] = __float2half_rn(__uint_as_float(v[j]));
            }
          } else {
            float* y = reinterpret_cast<float*>(p.y);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + cc + j;
              if (m < p.M && cc + j < p.BN) y[(size_t)m * p.N + n] = __uint_as_float(v[j]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, p.tmem_cols);
}

// ---------------------------------------------------------------- host --
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  *out = g_encode;
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t make_maps(const void* w0, const void* w1, const void* x, int64_t M, int64_t N, int64_t K, int BN,
                      CUtensorMap* mx, CUtensorMap* mw0, CUtensorMap* mw1) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {KSTEP, (cuuint32_t)BN};
    const cuuint32_t es[2] = {1, 1};
    if (enc(mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int64_t NB = K / QK;
  const cuuint64_t wdims[3] = {(cuuint64_t)BLOCK_BYTES, (cuuint64_t)NB, (cuuint64_t)N};
  const cuuint64_t wstrides[2] = {(cuuint64_t)BLOCK_BYTES, (cuuint64_t)(NB * BLOCK_BYTES)};
  const cuuint32_t wbox[3] = {BLOCK_BYTES, 1, TILE_N};
  const cuuint32_t wes[3] = {1, 1, 1};
  const void* ws[2] = {w0, w1 ? w1 : w0};
  CUtensorMap* maps[2] = {mw0, mw1};
  for (int i = 0; i < 2; ++i) {
    if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ws[i]), wdims, wstrides, wbox, wes,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <bool SWIGLU>
cudaError_t launch_tc(const CUtensorMap& mx, const CUtensorMap& mw0, const CUtensorMap& mw1, GemmParams p,
                      int64_t N, cudaStream_t s, size_t smem) {
  auto kern = q4k_gemm_tc_kernel<SWIGLU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((N + TILE_N - 1) / TILE_N), (unsigned)((p.M + p.BN - 1) / p.BN));
  kern<<<grid, 320, smem, s>>>(mx, mw0, mw1, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc(const void* w0, const void* w1, const void* x, void* y, bool y_f16, int64_t M,
                           int64_t N, int64_t K, cudaStream_t s) {
  const DevInfo& dev = device_info();
  const bool swiglu = w1 != nullptr;
  const int nmat = swiglu ? 2 : 1;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K / QK > INT32_MAX / 8) return cudaErrorInvalidValue;
  // Tokens per CTA: the whole of M up to 256 (rounded up to 16), else 256
  // (128 when the SwiGLU epilogue needs two accumulators).  Stage counts:
  // raw-W and dequantised-A rings first, the rest of shared memory for X.
  // JLLM_GEMM_BN / _SA / _SW override (tuning).
  static const int env_bn = getenv("JLLM_GEMM_BN") ? atoi(getenv("JLLM_GEMM_BN")) : 0;
  static const int env_sa = getenv("JLLM_GEMM_SA") ? atoi(getenv("JLLM_GEMM_SA")) : 0;
  static const int env_sw = getenv("JLLM_GEMM_SW") ? atoi(getenv("JLLM_GEMM_SW")) : 0;
  int bn_cap = swiglu ? 128 : 256;
  if (env_bn >= 16 && env_bn <= bn_cap && env_bn % 16 == 0) bn_cap = env_bn;
  int BN = (int)((M + 15) / 16 * 16);
  if (BN > bn_cap) BN = bn_cap;
  uint32_t cols = 32;
  while (cols < (uint32_t)(BN * nmat)) cols <<= 1;

  GemmParams p;
  p.y = y;
  p.M = (int)M;
  p.N = (int)N;
  p.NB = (int)(K / QK);
  p.BN = BN;
  p.tmem_cols = cols;
  p.out_f16 = (y_f16 || swiglu) ? 1 : 0;
  p.SW = env_sw > 0 ? env_sw : 3;
  p.SA = env_sa > 0 ? env_sa : 3;
  const size_t x_stage = (size_t)BN * KSTEP * 2;
  const size_t budget = dev.smem_optin - 1024 /*alignment*/ - 512 /*barriers*/;
  size_t fixed = (size_t)p.SW * W_STAGE_BYTES * nmat + (size_t)p.SA * A_STAGE_BYTES * nmat;
  while (fixed + 2 * x_stage > budget && (p.SW > 2 || p.SA > 2)) {
    if (p.SW >= p.SA && p.SW > 2) --p.SW; else --p.SA;
    fixed = (size_t)p.SW * W_STAGE_BYTES * nmat + (size_t)p.SA * A_STAGE_BYTES * nmat;
  }
  if (fixed + 2 * x_stage > budget) return cudaErrorInvalidValue;
  size_t sxn = (budget - fixed) / x_stage;
  if (sxn > 8) sxn = 8;
  p.SX = (int)sxn;
  p.off_x = 0;
  p.off_a = (uint32_t)(p.SX * x_stage);
  p.off_w = p.off_a + (uint32_t)(p.SA * A_STAGE_BYTES * nmat);
  p.off_bar = p.off_w + (uint32_t)(p.SW * W_STAGE_BYTES * nmat);
  const size_t smem = 1024 + p.off_bar + 8 * (2 * (p.SX + p.SW + p.SA) + 1) + 16;

  CUtensorMap mx, mw0, mw1;
  cudaError_t e = make_maps(w0, w1, x, M, N, K, BN, &mx, &mw0, &mw1);
  if (e != cudaSuccess) return e;
  return swiglu ? launch_tc<true>(mx, mw0, mw1, p, N, s, smem) : launch_tc<false>(mx, mw0, mw1, p, N, s, smem);
}

cudaError_t read_clear_gemm_error(uint32_t* bits, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

}  // namespace jllm

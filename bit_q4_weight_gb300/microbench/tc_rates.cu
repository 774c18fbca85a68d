// Tensor-core rate micro-benchmark: what an int8 ("MMQ") variant of the Q4_K
// prefill GEMM could use on this part.
//
//  * tcgen05.mma kind::f16 (fp16 x fp16 -> fp32, cta_group::1, M = 128,
//    N = 256, K-major 128-byte swizzle operands in shared memory): the path
//    the GEMM uses.  One CTA per SM; one thread issues `iters` groups of four
//    MMAs (a 128-byte K slice) on resident operands, commits and waits once.
//  * mma.sync m16n8k16 f16 -> f32 and m16n8k32 s8 -> s32 (the warp-level
//    tensor instructions): 8 warps per SM, each with 4 independent
//    accumulator chains on register operands.
//  * the tcgen05 stream as a pipelined GEMM issues it: a tcgen05.commit per
//    4-MMA step (onto a barrier nobody waits for) and one mbarrier probe per
//    step on a barrier whose phase has already completed -- none (kind 5),
//    mbarrier.try_wait (kind 3) or the non-blocking mbarrier.test_wait
//    (kind 4): what the issuer pays per stage even when its operands are ready.
// tcgen05.mma kind::i8 is not in the list: the CUDA 13.0 assembler rejects it
// for sm_103a ("Feature '.kind::i8' not supported on .target 'sm_103a'").
// Operands are zeros, so the values play no part.  Not part of the Q4_K
// library: bench.py builds it into its own shared object for --tc-rates.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../csrc/common.cuh"

namespace {

constexpr int TM = 128, TN = 256;
constexpr int A_BYTES = TM * 128, B_BYTES = TN * 128;  // one 128-byte K slice each
constexpr uint64_t LIMIT_NS = 2000000000ull;

__device__ uint32_t g_tc_error;

// PROBE: 0 plain stream; 3 commit + try_wait, 4 commit + test_wait, 5 commit
// alone, per 4-MMA step.
template <int PROBE>
__global__ void __launch_bounds__(128, 1) tcgen05_f16_kernel(int iters, unsigned long long* cycles) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar, done_bar, step_bar;
  __shared__ uint32_t tmem_slot;
  for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    jllm::mbar_init(jllm::smem_u32(&bar), 1);
    jllm::mbar_init(jllm::smem_u32(&done_bar), 1);
    jllm::mbar_init(jllm::smem_u32(&step_bar), 1);
    jllm::fence_mbarrier_init();
    jllm::mbar_arrive(jllm::smem_u32(&done_bar));  // its phase 0 is complete from here on
  }
  if (warp == 0) jllm::tmem_alloc(jllm::smem_u32(&tmem_slot), TN);
  jllm::fence_proxy_async_smem();  // the zero fill, visible to the tensor core
  jllm::tc_fence_before();
  __syncthreads();
  jllm::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) {
    const uint32_t sa = jllm::smem_u32(smem), sb = sa + A_BYTES;
    const uint64_t ad = jllm::umma_desc_sw128(sa), bd = jllm::umma_desc_sw128(sb);
    const uint32_t idesc = jllm::umma_idesc_f16(TM, TN);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      if (PROBE == 3 && !jllm::mbar_try_wait(jllm::smem_u32(&done_bar), 0)) atomicOr(&g_tc_error, 2u);
      if (PROBE == 4 && !jllm::mbar_test_wait(jllm::smem_u32(&done_bar), 0)) atomicOr(&g_tc_error, 2u);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) jllm::umma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (it | kk) ? 1u : 0u);
      if (PROBE != 0) jllm::umma_commit(jllm::smem_u32(&step_bar));
    }
    jllm::umma_commit(jllm::smem_u32(&bar));
    if (!jllm::mbar_wait_bounded(jllm::smem_u32(&bar), 0, nullptr, LIMIT_NS)) atomicOr(&g_tc_error, 1u);
    cycles[blockIdx.x] = (unsigned long long)(clock64() - t0);
  }
  jllm::tc_fence_before();
  __syncthreads();
  jllm::tc_fence_after();
  if (warp == 0) jllm::tmem_dealloc(tmem, TN);
}

// 4 independent m16n8k16 f16 -> f32 (or m16n8k32 s8 -> s32) chains per warp.
template <bool S8>
__global__ void __launch_bounds__(256) mma_sync_kernel(int iters, unsigned long long* cycles, int* sink) {
  uint32_t a[4] = {0u, 0u, 0u, 0u}, b[2] = {0u, 0u};
  uint32_t d[4][4] = {};
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (S8)
        asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
      else
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
  }
  const long long t1 = clock64();
  if ((threadIdx.x & 31) == 0) cycles[blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)] = (unsigned long long)(t1 - t0);
  int acc = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) acc ^= (int)(d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3]);
  if (acc == 12345) sink[0] = acc;  // keeps the chains live
}

}  // namespace

// kind = 0: tcgen05 kind::f16, one CTA (one issuing thread) per block, cycles_dev[ctas];
// kind = 1: mma.sync f16, kind = 2: mma.sync s8, 8 warps per block, cycles_dev[ctas * 8];
// kind = 3 / 4 / 5: kind 0 with a commit and an mbarrier.try_wait / test_wait /
// no probe per 4 MMAs.
// Synchronises `stream`.  Returns a cudaError_t value, or 1000 + n when n
// bounded waits ran out.
extern "C" int jllm_microbench_tc_rate(int kind, int ctas, int iters, unsigned long long* cycles_dev, int* sink,
                                       void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (kind == 0 || kind == 3 || kind == 4 || kind == 5) {
    const size_t smem = (size_t)A_BYTES + B_BYTES + 1024;
    auto kern = kind == 0 ? tcgen05_f16_kernel<0>
                : kind == 3 ? tcgen05_f16_kernel<3>
                : kind == 4 ? tcgen05_f16_kernel<4> : tcgen05_f16_kernel<5>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) kern<<<ctas, 128, smem, s>>>(iters, cycles_dev);
  } else if (kind == 1) {
    mma_sync_kernel<false><<<ctas, 256, 0, s>>>(iters, cycles_dev, sink);
  } else if (kind == 2) {
    mma_sync_kernel<true><<<ctas, 256, 0, s>>>(iters, cycles_dev, sink);
  } else {
    return (int)cudaErrorInvalidValue;
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return (int)e;
  uint32_t bad = 0;
  e = cudaMemcpyFromSymbol(&bad, g_tc_error, sizeof(bad));
  if (e != cudaSuccess) return (int)e;
  return bad ? 1000 + (int)bad : 0;
}

// Q4_K GEMV chain: a sequence of dependent one-token GEMV steps (a decode
// step's q/k/v, o, gate/up, down projections, layer after layer) in ONE
// persistent launch.
//
// The decode kernel of the genie-ai-runtime README ("At a glance", Kernels
// bullet: "INT4 dequant-fused GEMV"), as a whole-sweep kernel for sm_103a.
// One launch per matmul leaves a fixed cost per launch on the critical path
// (the previous launch's tail and completion, x staging behind the next
// launch's weight copies, few warps per SM on the small matrices); here:
//
//  * One CTA per SM (cooperative launch: all resident), 16 compute warps and
//    one producer warp.  The producer streams the CTA's weight rows of every
//    step, in step order, HBM -> shared memory by cp.async.bulk into a ring of
//    four 46 KiB slots -- independently of the steps' data dependences, so
//    the HBM keeps streaming while the compute warps wait for the previous
//    step's results.
//  * Step s's rows (its matrices concatenated) are split evenly over the
//    CTAs; a CTA's rows are cut at matrix boundaries into chunks of whole
//    rows (at most one slot, at most 64 rows).  A chunk's (row, block pair)
//    units are split evenly over the 64 eight-lane groups, so a group may
//    take part of a row (split K): its partial row sums go to shared memory
//    and one thread per row adds them in group order (deterministic).
//  * Dependences: after its last y write of step s, a CTA counts itself in
//    the step's counter (release); before staging x of step s+1, it waits
//    until the counter reaches the grid size (acquire).  The last CTA to
//    finish the launch returns the counters to zero.
//  * The inner product and the x staging are those of the per-launch GEMV
//    (q4k_dot.cuh): fp16 subnormal codes, exact products, fp32 sums.
// Every wait is bounded: a wait that runs out sets the device error word and
// the CTA winds down (copies in flight awaited); the counters are then left
// as they were and must be zeroed again by the caller.
#include "common.cuh"
#include "internal.h"
#include "q4k_dot.cuh"

namespace jllm {

__device__ uint32_t g_chain_error;

namespace {

#ifndef JLLM_WAIT_LIMIT_NS
#define JLLM_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t CHAIN_WAIT_LIMIT_NS = JLLM_WAIT_LIMIT_NS;  // 2 s (a test build shortens it)

#ifdef JLLM_FAULT_INJECTION
// Test builds only: when set, CTA 0's producer never issues its first copy,
// so the compute warps' bounded wait runs out and the timeout path runs.
__device__ int g_fi_skip_chain;
#endif

constexpr int CH_WARPS = 16;                        // compute warps
constexpr int CH_CTHREADS = CH_WARPS * 32;          // compute threads (named barrier 1)
constexpr int CH_THREADS = CH_CTHREADS + 32;        // + the producer warp
constexpr int CH_GROUPS = CH_WARPS * 4;             // eight-lane groups
constexpr int CH_SLOTS = 4;
constexpr uint32_t CH_SLOT_BYTES = 46 * 1024;       // a multiple of 16
constexpr int CH_MAX_ROWS = 64;                     // rows per chunk (a group then spans <= 2 rows)
constexpr int CH_PART_CHUNKS = CH_CTHREADS / CH_MAX_ROWS;  // chunks reduced together (one thread per row)

// Shared-memory carve-up (bytes).
constexpr uint32_t OFF_SLOTS = 0;
constexpr uint32_t OFF_XS = OFF_SLOTS + CH_SLOTS * CH_SLOT_BYTES;
constexpr uint32_t OFF_XSUM = OFF_XS + kChainMaxBlocks * 36 * 16;
constexpr uint32_t OFF_PART = OFF_XSUM + kChainMaxBlocks * 8 * 4;
constexpr uint32_t OFF_META = OFF_PART + CH_PART_CHUNKS * CH_GROUPS * 2 * 4;
constexpr uint32_t OFF_BARS = OFF_META + CH_PART_CHUNKS * 16;
constexpr uint32_t OFF_FLAG = OFF_BARS + 2 * CH_SLOTS * 8;
constexpr uint32_t CH_SMEM = OFF_FLAG + 16;

static_assert(kChainMaxSteps == JLLM_CHAIN_MAX_STEPS && kChainMaxMats == JLLM_CHAIN_MAX_MATS &&
                  kChainMaxBlocks * QK == JLLM_CHAIN_MAX_K,
              "chain limits of the C ABI");

struct ChainStep {
  const uint8_t* w[kChainMaxMats];  // [n][nb] blocks
  void* y[kChainMaxMats];           // [n] fp32, or fp16 when out_f16
  const __half* x;                  // [nb * 256] fp16
  int n[kChainMaxMats];
  int nb;                           // blocks per row (K / 256)
  int count;                        // matrices
  int rows;                         // sum of n
  int out_f16;
};

struct ChainParams {
  uint32_t* sync;  // [n_steps] step counters, then the exit counter
  int n_steps;
  int pad;
  ChainStep step[kChainMaxSteps];
};

__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_add_release_gpu_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acqrel_gpu_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Barrier over the compute warps that also returns the OR of `pred` over them,
// so that a failure seen by any thread is seen by all at the same point.
__device__ __forceinline__ bool compute_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "n"(CH_CTHREADS)
      : "memory");
  return r != 0;
}

// L2-coherent 16-byte load: x may have been written during this launch by
// another CTA, so the non-coherent path is not used.
__device__ __forceinline__ uint4 ldg_cg(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// This CTA's rows [r0, r1) of a step's concatenated rows.
__device__ __forceinline__ void cta_rows(int rows, int cta, int G, int& r0, int& r1) {
  r0 = (int)((int64_t)rows * cta / G);
  r1 = (int)((int64_t)rows * (cta + 1) / G);
}

// Walks the chunks of this CTA's rows of one step: matrix index, first local
// row and row count of each, in order.
struct ChunkWalk {
  int a, b;        // remaining concatenated rows [a, b)
  int mi, base;    // current matrix and its first concatenated row
  int seg_end, nseg, nch, ich, seg0;
  int maxr;
  __device__ void init(const ChainStep& st, int cta, int G) {
    cta_rows(st.rows, cta, G, a, b);
    mi = 0;
    base = 0;
    nch = 0;
    ich = 0;
    const int rb = st.nb * BLOCK_BYTES;
    maxr = (int)(CH_SLOT_BYTES / (uint32_t)rb);
    if (maxr > CH_MAX_ROWS) maxr = CH_MAX_ROWS;
  }
  // Next chunk; false when the CTA's rows of the step are done.
  __device__ bool next(const ChainStep& st, int& m, int& lrow0, int& nrows) {
    if (ich == nch) {
      if (a >= b) return false;
      while (a >= base + st.n[mi]) {
        base += st.n[mi];
        ++mi;
      }
      seg_end = min(b, base + st.n[mi]);
      seg0 = a;
      nseg = seg_end - a;
      nch = (nseg + maxr - 1) / maxr;
      ich = 0;
      a = seg_end;
    }
    const int c0 = seg0 + (int)((int64_t)nseg * ich / nch), c1 = seg0 + (int)((int64_t)nseg * (ich + 1) / nch);
    ++ich;
    m = mi;
    lrow0 = c0 - base;
    nrows = c1 - c0;
    return true;
  }
};

__device__ __forceinline__ const uint8_t* mat_w(const ChainStep& st, int m) {
  const uint8_t* w = st.w[0];
#pragma unroll
  for (int i = 1; i < kChainMaxMats; ++i)
    if (m == i) w = st.w[i];
  return w;
}
__device__ __forceinline__ void* mat_y(const ChainStep& st, int m) {
  void* y = st.y[0];
#pragma unroll
  for (int i = 1; i < kChainMaxMats; ++i)
    if (m == i) y = st.y[i];
  return y;
}

__global__ void __launch_bounds__(CH_THREADS, 1) q4k_gemv_chain_kernel(const __grid_constant__ ChainParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t b_full = sbase + OFF_BARS, b_empty = b_full + 8 * CH_SLOTS;
  uint4* xs = reinterpret_cast<uint4*>(smem + OFF_XS);
  float* Xs = reinterpret_cast<float*>(smem + OFF_XSUM);
  float* part = reinterpret_cast<float*>(smem + OFF_PART);  // [CH_PART_CHUNKS][CH_GROUPS][2]
  int4* meta = reinterpret_cast<int4*>(smem + OFF_META);     // (matrix, first row, rows, units) per chunk
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_FLAG);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (int)gridDim.x, cta = (int)blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < CH_SLOTS; ++i) {
      mbar_init(b_full + 8 * i, 1);
      mbar_init(b_empty + 8 * i, CH_WARPS);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == CH_WARPS) {
    // ------------------------------------------------------------ producer --
    if (lane != 0) return;
    const uint64_t pol = l2_policy_evict_first();  // weights are read once per call
    int slot = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    for (int s = 0; ok && s < p.n_steps; ++s) {
      const ChainStep& st = p.step[s];
      const int64_t rb = (int64_t)st.nb * BLOCK_BYTES;
      ChunkWalk cw;
      cw.init(st, cta, G);
      int m, l0, nr;
      while (cw.next(st, m, l0, nr)) {
        if (!mbar_wait_bounded(b_empty + 8 * slot, ph ^ 1u, abort_flag, CHAIN_WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t bytes = (uint32_t)(nr * rb);
#ifdef JLLM_FAULT_INJECTION
        if (!(issued == 0 && cta == 0 && g_fi_skip_chain))
#endif
        {
          mbar_arrive_expect_tx(b_full + 8 * slot, bytes);
          bulk_load_hint(sbase + OFF_SLOTS + (uint32_t)slot * CH_SLOT_BYTES, mat_w(st, m) + (int64_t)l0 * rb, bytes,
                         b_full + 8 * slot, pol);
        }
        ++issued;
        if (++slot == CH_SLOTS) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(&g_chain_error, ERR_TIMEOUT);
    }
    // Every copy issued must have landed before the CTA exits (the compute
    // warps consume them all on the normal path; after a failure they may not).
    if (*abort_flag) {
      for (long long i = issued > CH_SLOTS ? issued - CH_SLOTS : 0; i < issued; ++i)
        mbar_wait_bounded(b_full + 8 * (int)(i % CH_SLOTS), (uint32_t)((i / CH_SLOTS) & 1), nullptr,
                          CHAIN_WAIT_LIMIT_NS);
    }
    return;
  }

  // -------------------------------------------------------------- compute --
  const int tid = threadIdx.x;
  const int grp = lane >> 3, t = lane & 7, kp = t >> 2, c = t & 3;
  const int gi = warp * 4 + grp;
  const unsigned gmask = 0xFFu << (8 * grp);
  const LaneDec L = lane_dec(c);
  int slot = 0;
  uint32_t ph = 0;
  bool fail = false;
  pdl_wait();  // x, y and the counters are touched only after the previous kernel

  for (int s = 0; s < p.n_steps; ++s) {
    const ChainStep& st = p.step[s];
    const int nb = st.nb;
    const int rb = nb * BLOCK_BYTES;
    const int nb2 = (nb + 1) >> 1;
    // The previous step's y is complete everywhere once its counter reaches G.
    if (s > 0 && tid == 0) {
      const uint32_t* cnt = p.sync + (s - 1);
      if (ld_acquire_gpu_u32(cnt) < (uint32_t)G) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
          if (ld_acquire_gpu_u32(cnt) >= (uint32_t)G) break;
          if ((it & 63u) == 0 && (*abort_flag || globaltimer_ns() - t0 > CHAIN_WAIT_LIMIT_NS)) {
            fail = true;
            break;
          }
        }
      }
    }
    if (compute_sync_or(fail)) {
      fail = true;
      break;
    }
    // Stage x: one 32-element sub-block per thread (nb * 8 <= 512), padded
    // layout and the sums X_j * 2^-24.
    if (tid < nb * 8) {
      const int kr = tid >> 3, j = tid & 7;
      const __half* src = st.x + (size_t)tid * 32;
      uint4 u[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) u[v] = ldg_cg(src + 8 * v);
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        xs[x_unit_pos(kr, j >> 1, 4 * (j & 1) + v)] = u[v];
        add_halves(s4[v], u[v].x);
        add_halves(s4[v], u[v].y);
        add_halves(s4[v], u[v].z);
        add_halves(s4[v], u[v].w);
      }
      Xs[tid] = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * kTwoM24;
    }
    compute_sync_or(false);

    ChunkWalk cw;
    cw.init(st, cta, G);
    int m, l0, nr;
    bool more = cw.next(st, m, l0, nr);
    int nck = 0;  // chunks whose partial sums wait in part[]
    while (more) {
      const int U = nr * nb2;
      const int u0 = (int)((int64_t)U * gi / CH_GROUPS), u1 = (int)((int64_t)U * (gi + 1) / CH_GROUPS);
      float* pg = part + (nck * CH_GROUPS + gi) * 2;
      if (tid == 0) meta[nck] = make_int4(m, l0, nr, U);
      const bool have = mbar_wait_warp(b_full + 8 * slot, ph, abort_flag, CHAIN_WAIT_LIMIT_NS);
      if (!have) {
        fail = true;
        *abort_flag = 1;
      } else if (u0 == u1) {
        if (t == 0) pg[0] = 0.f;  // an empty group adds an exact zero to the row it falls in
      } else {
        const uint8_t* chunk = smem + OFF_SLOTS + (size_t)slot * CH_SLOT_BYTES;
        float acc = 0.f;
        int row = u0 / nb2, jrow = 0;
        int pr = u0 - row * nb2;
        for (int u = u0; u < u1; ++u) {
          const int kr = 2 * pr + kp;
          if (kr < nb) {
            const uint8_t* blk = chunk + (size_t)row * rb + kr * BLOCK_BYTES;
            RowData d;
            d.h = *reinterpret_cast<const uint4*>(blk);
            d.q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
            d.q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
            uint4 xv[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) xv[b] = xs[x_unit_pos(kr, c, b)];
            const float2 X = *reinterpret_cast<const float2*>(&Xs[kr * 8 + 2 * c]);
            chunk_dot(acc, d, xv, X.x, X.y, L);
          }
          if (++pr == nb2 || u + 1 == u1) {  // the group's part of this row is done
            float v = acc;
            v += __shfl_xor_sync(gmask, v, 1);
            v += __shfl_xor_sync(gmask, v, 2);
            v += __shfl_xor_sync(gmask, v, 4);
            if (t == 0) pg[jrow] = v;
            acc = 0.f;
            pr = 0;
            ++row;
            ++jrow;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(b_empty + 8 * slot);
      if (++slot == CH_SLOTS) {
        slot = 0;
        ph ^= 1u;
      }
      ++nck;
      more = cw.next(st, m, l0, nr);
      if (nck < CH_PART_CHUNKS && more) continue;
      // Row sums of the buffered chunks, one thread per (chunk, row): the groups
      // whose unit ranges meet row r are a contiguous range, added in order.
      if (compute_sync_or(fail)) {
        fail = true;
        break;
      }
      {
        const int ck = tid >> 6, r = tid & 63;
        if (ck < nck) {
          const int4 md = meta[ck];
          if (r < md.z) {
            const int Uc = md.w;
            const int ua = r * nb2, uz = ua + nb2 - 1;                // first and last unit of row r
            const int ga = (CH_GROUPS * (ua + 1) - 1) / Uc, gz = (CH_GROUPS * (uz + 1) - 1) / Uc;
            const float* pc = part + ck * CH_GROUPS * 2;
            // group ga holds row r in slot 1 when its range began in row r-1
            float sum = pc[ga * 2 + (((int64_t)Uc * ga / CH_GROUPS) < ua ? 1 : 0)];
            for (int g = ga + 1; g <= gz; ++g) sum += pc[g * 2];
            if (st.out_f16) static_cast<__half*>(mat_y(st, md.x))[md.y + r] = __float2half_rn(sum * kTwo24);
            else static_cast<float*>(mat_y(st, md.x))[md.y + r] = sum * kTwo24;
          }
        }
      }
      nck = 0;
      if (more && compute_sync_or(fail)) {  // part[] and meta[] are reused
        fail = true;
        break;
      }
    }
    if (compute_sync_or(fail)) {
      fail = true;
      break;
    }
    if (tid == 0) red_add_release_gpu_u32(p.sync + s, 1u);
  }

  if (fail) {
    if (tid == 0) {
      *abort_flag = 1;
      atomicOr(&g_chain_error, ERR_TIMEOUT);
    }
    return;
  }
  // The last CTA out returns the counters to zero for the next launch.
  if (tid == 0) {
    __threadfence();
    if (atom_add_acqrel_gpu_u32(p.sync + p.n_steps, 1u) == (uint32_t)(G - 1)) {
      for (int s = 0; s <= p.n_steps; ++s) p.sync[s] = 0u;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_gemv_chain(const jllm_gemv_step* steps, int n_steps, uint32_t* sync, cudaStream_t stream) {
  if (n_steps < 1 || n_steps > kChainMaxSteps || steps == nullptr || sync == nullptr ||
      (reinterpret_cast<uintptr_t>(sync) & 3u))
    return cudaErrorInvalidValue;
  static_assert(sizeof(ChainParams) <= 32000, "kernel parameter space");
  // Large (26 KiB): kept off the stack, one per host thread; the launch copies it.
  thread_local ChainParams P;
  P = ChainParams{};
  P.sync = sync;
  P.n_steps = n_steps;
  for (int s = 0; s < n_steps; ++s) {
    const jllm_gemv_step& d = steps[s];
    ChainStep& st = P.step[s];
    if (d.count < 1 || d.count > kChainMaxMats || d.K <= 0 || d.K % QK || d.K / QK > kChainMaxBlocks ||
        d.x == nullptr || (reinterpret_cast<uintptr_t>(d.x) & 15u) || (d.y_f16 != 0 && d.y_f16 != 1))
      return cudaErrorInvalidValue;
    int64_t rows = 0;
    for (int i = 0; i < d.count; ++i) {
      if (d.N[i] < 0 || d.N[i] > INT32_MAX || (d.N[i] > 0 && (d.w_q4k[i] == nullptr || d.y[i] == nullptr)) ||
          (reinterpret_cast<uintptr_t>(d.w_q4k[i]) & 15u) || (reinterpret_cast<uintptr_t>(d.y[i]) & 3u))
        return cudaErrorInvalidValue;
      st.w[i] = static_cast<const uint8_t*>(d.w_q4k[i]);
      st.y[i] = d.y[i];
      st.n[i] = (int)d.N[i];
      rows += d.N[i];
    }
    if (rows > INT32_MAX) return cudaErrorInvalidValue;
    st.x = static_cast<const __half*>(d.x);
    st.nb = (int)(d.K / QK);
    st.count = d.count;
    st.rows = (int)rows;
    st.out_f16 = d.y_f16;
  }
  const DevInfo& dev = device_info();
  if (dev.err != cudaSuccess) return dev.err;
  cudaError_t e = cudaFuncSetAttribute(q4k_gemv_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CH_SMEM);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q4k_gemv_chain_kernel, CH_THREADS, CH_SMEM);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)dev.sm_count);
  cfg.blockDim = dim3(CH_THREADS);
  cfg.dynamicSmemBytes = CH_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  attr[na].id = cudaLaunchAttributeCooperative;  // the CTAs wait on one another's step counters
  attr[na].val.cooperative = 1;
  ++na;
  if (dev.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, q4k_gemv_chain_kernel, P);
}

#ifdef JLLM_FAULT_INJECTION
cudaError_t fault_injection_set_chain(int skip) { return cudaMemcpyToSymbol(g_fi_skip_chain, &skip, sizeof(int)); }
#endif

cudaError_t read_clear_chain_error(uint32_t* bits) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_chain_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_chain_error, &z, sizeof(z));
  }
  *bits = v;
  return e;
}

}  // namespace jllm

// Q4_K dequant-fused GEMM on the sm_103a tensor cores: Y = X * dequant(W)^T.
//
// The prefill kernel of the genie-ai-runtime README ("At a glance", Kernels
// bullet: "tensor-core MMQ Q4_K prefill"), re-designed around TMA, tcgen05
// and tensor memory.
//
// Orientation.  The MMA computes D[128 weight rows][BN tokens] += A * B^T with
// A = the dequantised fp16 weight tile (M = 128 rows of W, K-major) and B = a
// tile of X (N = BN tokens, K-major).  Putting W on the MMA's M side means a
// weight is dequantised once per tile and reused for BN tokens.  D lives in
// tensor memory (lane = weight row, column = token, fp32).
//
// Persistent schedule.  One CTA per SM walks a contiguous range of "units":
// the K steps (64 wide, 128 with A in tensor memory) of the tiles laid out
// tile after tile.  Without a workspace a range is a whole number of tiles.
// With one (stream-K), the ranges are equal in K steps, so the last wave of
// tiles is shared out evenly; a tile cut between CTAs is finished by the CTA
// that owns its first K step, which adds the fp32 partial sums the later CTAs
// left in the workspace, in CTA order (deterministic).  Tiles of at most 128
// tokens that number at most a quarter of the SMs are split instead over a
// thread-block cluster of 4-8 CTAs per tile (cluster split-K): each CTA takes
// an equal share of the tile's K steps, and the partials are added in K order
// through distributed shared memory.
//
// Roles (448 threads):
//   warp 0      TMA producer: per K step one X tile {64 k x BN tokens},
//               128-byte swizzled; per 256-wide block one raw W tile
//               {144 bytes x 1 block x 128 rows} through a 3-D byte view.
//   warp 1      TMEM owner (512 columns = two accumulator buffers, or one
//               for tiles of more than 256 tokens) and MMA issuer (one
//               thread): four tcgen05.mma (K = 16) per K step and token half,
//               tcgen05.commit frees the stages and, per unit, hands the
//               accumulator buffer to the epilogue.
//   warps 2-9   dequantisers, two threads per weight row (low / high nibbles
//               of the row's 32 code bytes for the step): the values
//               (d*sc)*q - dmin*m exactly as the fp32 dequant forms them,
//               rounded to fp16, stored in the 128-byte-swizzle K-major
//               layout the MMA descriptor reads.
//   warps 10-13 epilogue: tcgen05.ld of one TMEM lane quarter, store Y
//               (fp32 / fp16) or silu(g)*u (fp16), or the fp32 partial of a
//               cut tile.  It runs while the MMA fills the other buffer (or,
//               with one buffer, the half already drained).
// Ring positions advance by counters (stage, phase), never by division.
// Programmatic dependent launch: setup and the first weight blocks overlap
// the previous kernel in the stream; X is loaded and Y, the partials and the
// flags are written only after griddepcontrol.wait.
// Every wait is bounded; a wait that runs out sets the device error word
// and the CTA winds down (copies and MMAs in flight are awaited, TMEM is
// freed).
#include <cudaTypedefs.h>

#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace jllm {
namespace {

__device__ uint32_t g_gemm_error;

#ifdef JLLM_FAULT_INJECTION
// Test builds only: when set, the producer of CTA 0 never issues its first X
// copy, so the MMA warp's bounded wait on that stage runs out and the whole
// timeout path runs (error word, abort flag, wind-down, TMEM freed).
__device__ int g_fi_skip_x;
#endif

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

// Cluster split-K: remote arrive on the same barrier in another CTA of the
// cluster, a bounded wait that acquires at cluster scope, and a load from
// another CTA's shared memory.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint32_t atom_add_acqrel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

constexpr int TILE_N = 128;                         // weight rows per tile (MMA M)
constexpr int KSTEP = 64;                           // K per stage (128 bytes of fp16)
constexpr int A_STAGE_BYTES = TILE_N * KSTEP * 2;   // 16 KiB
constexpr int W_STAGE_BYTES = TILE_N * BLOCK_BYTES; // 18 KiB
constexpr int NUM_THREADS = 448;
constexpr int EPI_WARP0 = 10;                       // warps 10..13
constexpr int NUM_EPI_WARPS = 4;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;                  // TMEM columns per accumulator buffer
constexpr int SLOT_FLOATS = TILE_N * 512;           // fp32 partial of one tile (256 KiB)
#ifndef JLLM_WAIT_LIMIT_NS
#define JLLM_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t WAIT_LIMIT_NS = JLLM_WAIT_LIMIT_NS;  // 2 s (a test build shortens it)

// ATMEM: the dequantised weight tile (the MMA's A operand) is written to
// tensor memory with tcgen05.st instead of shared memory, so the tensor core
// reads only X from shared memory.  Tensor memory then holds two accumulators
// of at most ACC_COLS_ATMEM columns and SA A stages of 32 columns (128 rows x
// 64 fp16, two per 32-bit column).
constexpr uint32_t ACC_COLS_ATMEM = 128;
constexpr uint32_t A_TMEM_COL0 = 2 * ACC_COLS_ATMEM;  // first column of the A ring

// WIDE: tiles of up to 512 tokens for long prompts.  Each K = 16 slice takes
// two MMAs of BN/2 tokens (the two halves of the X stage) into one accumulator
// of all 512 tensor-memory columns (half h at column 256*h), so a dequantised
// weight meets twice the tokens per synchronisation round.  The epilogue
// releases the halves one at a time, and the next tile's first MMAs into half
// 0 start while half 1 is still being drained.
// SWIGLU: the tile's 128 rows pair 64 gate with 64 up rows (in each 32-lane
// quarter of tensor memory, lanes 0-15 gate and 16-31 the up rows of the same
// outputs), and the epilogue writes h = silu(g) * u for 64 outputs per tile;
// otherwise the same kernel.
template <bool SWIGLU, bool ATMEM = false, bool WIDE = false>
struct Cfg {
  static constexpr int NMAT = 1;                         // raw-W / A stages per K step
  // K per pipeline step: 128 with A in tensor memory (two 64-wide X boxes and
  // eight MMAs per synchronisation round), else 64 (one 128-byte swizzle atom
  // of the A tile in shared memory).
  static constexpr int KST = ATMEM ? 128 : KSTEP;
  static constexpr int SPB = QK / KST;                   // steps per super-block
  static constexpr uint32_t ASC = KST / 2;               // tensor-memory columns of an A stage
  static constexpr int SX = ATMEM ? 4 : (WIDE ? 2 : 3);  // X ring
  // COMB: X and A share one stage index, one full barrier (the X copy and the 8
  // dequant warps arrive on it) and one empty barrier (one commit per K step).
  // Taken with A in tensor memory, where the A ring can match the X ring; with A
  // in shared memory the shorter A ring it would need costs more than it saves.
  static constexpr bool COMB = ATMEM;
  static constexpr int SA = COMB ? SX : (WIDE ? 3 : 4);  // dequantised-A ring
  static constexpr int SW = WIDE ? 2 : 3;                // raw-W ring
  static constexpr int XH = WIDE ? 2 : 1;                // token halves (X boxes, MMAs) per K slice
  // X ring slots: a stage, or (wide tiles) one token half of a stage, each with
  // its own full / empty barrier, so that a half's MMAs start when its box has
  // landed and its box is refilled as soon as they are done.
  static constexpr int XS = SX * XH;
  static constexpr int NACC = WIDE ? 1 : 2;              // accumulator buffers
  static constexpr int BN_MAX = ATMEM ? (int)ACC_COLS_ATMEM : (WIDE ? 512 : 256);
  static constexpr uint32_t ACC = ATMEM ? ACC_COLS_ATMEM : (WIDE ? TMEM_COLS : ACC_COLS);  // TMEM columns per accumulator
  static constexpr int NBARS = 2 * (XS + SA + SW) + 2 + 2 + 1 + 1;
  static_assert(!ATMEM || A_TMEM_COL0 + SA * ASC <= TMEM_COLS, "tensor memory budget");
  static_assert(!WIDE || !ATMEM, "wide tiles: A in shared memory");
  static_assert(BN_MAX % 16 == 0, "token tiles are multiples of 16");
};

// Up to kMaxGemmBatch weight matrices that share X (and so K) run in one
// launch: matrix b owns tiles [tile0[b], tile0[b+1]) of the tile space.
constexpr int kBatchMax = kMaxGemmBatch;

struct GemmParams {
  void* y[kBatchMax];    // [M][N[b]] fp32 / fp16 (h for SwiGLU)
  int N[kBatchMax];
  int tile0[kBatchMax + 1];
  int count;             // matrices in the batch (1 with SwiGLU: gate/up feed one output)
  float* partial;        // stream-K slots, SLOT_FLOATS per CTA (nullptr: whole tiles only)
  uint32_t* flags;       // one counter per CTA next to the slots
  int M, NB;
  int BN;                // tokens per tile, multiple of 16 (of 64 for wide tiles)
  int HB;                // tokens per MMA and X box: BN, or BN / 2 for wide tiles
  int m_tiles;           // ceil(M / BN)
  int KS;                // K steps per tile (4 per super-block)
  long long grains;      // units / grain
  int grain;             // KS (whole tiles) or 1 (stream-K)
  uint32_t x_stage_bytes;
  uint32_t off_x, off_a, off_w, off_bar;
  int out_f16;
  int csk;               // cluster split-K: CTAs per tile (a cluster), 0 = ranges over the tile list
  int pair;              // SwiGLU: a tile's 128 rows interleave 64 gate and 64 up rows, Y = silu(g)*u
};

// Stage index and phase parity of a ring of S stages.
template <int S>
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Tensor maps of the weight matrices: one per batch entry, or gate and up.
struct WMaps {
  CUtensorMap w[kBatchMax];
};

// Batch entry, output row and token of a tile; with all index reads on
// constant offsets of the parameter block.
struct TileLoc {
  int b, n0, m0, N;
  void* y;
};
__device__ __forceinline__ TileLoc locate(const GemmParams& p, int tile) {
  TileLoc t;
  t.b = 0;
  t.N = p.N[0];
  t.y = p.y[0];
  int base = 0;
#pragma unroll
  for (int i = 1; i < kBatchMax; ++i)
    if (i < p.count && tile >= p.tile0[i]) {
      t.b = i;
      t.N = p.N[i];
      t.y = p.y[i];
      base = p.tile0[i];
    }
  const int local = tile - base;
  const int nt = local / p.m_tiles;
  t.n0 = nt * (p.pair ? TILE_N / 2 : TILE_N);  // output columns: 64 per tile in SwiGLU pairs
  t.m0 = (local - nt * p.m_tiles) * p.BN;
  return t;
}

__device__ __forceinline__ long long range_start(const GemmParams& p, long long g) {
  return (g * p.grains / gridDim.x) * p.grain;
}

// Walks the units of one CTA's range: tile, and its K steps [k0, k1).
struct UnitIter {
  long long u, end;
  int KS;
  int tile = 0, k0 = 0, k1 = 0;
  __device__ __forceinline__ bool next() {
    if (u >= end) return false;
    tile = (int)(u / KS);
    k0 = (int)(u - (long long)tile * KS);
    const long long rem = end - u;
    k1 = rem < (long long)(KS - k0) ? k0 + (int)rem : KS;
    u += k1 - k0;
    return true;
  }
};

// acc += A * B^T with A (128 x 16 fp16) in tensor memory at column a_tmem.
__device__ __forceinline__ void umma_f16_ta(uint32_t tmem_d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 columns of 32-bit words: thread i of the warp writes lane
// (base lane + i), columns col..col+15.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
      " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <bool SWIGLU, bool ATMEM, bool WIDE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    q4k_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ WMaps tmW,
                       const __grid_constant__ GemmParams p) {
  using C = Cfg<SWIGLU, ATMEM, WIDE>;
  constexpr int NMAT = C::NMAT, SA = C::SA, SW = C::SW, XS = C::XS;
  extern __shared__ uint8_t gemm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sx = sbase + p.off_x, sa = sbase + p.off_a, sw = sbase + p.off_w;
  // barriers: x_full[XS] x_empty[XS] a_full[SA] a_empty[SA] w_full[SW] w_empty[SW]
  //           (COMB: x_full / x_empty serve X and A; a_full / a_empty unused)
  //           acc_full[2] acc_empty[2] drain cluster_ready
  const uint32_t b_xfull = sbase + p.off_bar, b_xempty = b_xfull + 8 * XS;
  const uint32_t b_afull = b_xempty + 8 * XS, b_aempty = b_afull + 8 * SA;
  const uint32_t x_slot_bytes = p.x_stage_bytes / C::XH;  // X ring slot: a stage or half of one
  const uint32_t b_wfull = b_aempty + 8 * SA, b_wempty = b_wfull + 8 * SW;
  const uint32_t b_accfull = b_wempty + 8 * SW, b_accempty = b_accfull + 16, b_drain = b_accempty + 16;
  const uint32_t b_cready = b_drain + 8;  // cluster split-K: the partials of the cluster are in place
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.off_bar + 8 * C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < XS; ++i) {
      mbar_init(b_xfull + 8 * i, C::COMB ? 9 : 1);  // COMB: the X copy and the 8 dequant warps
      mbar_init(b_xempty + 8 * i, 1);
    }
    for (int i = 0; i < SA; ++i) {
      mbar_init(b_afull + 8 * i, 8);
      mbar_init(b_aempty + 8 * i, 1);
    }
    for (int i = 0; i < SW; ++i) {
      mbar_init(b_wfull + 8 * i, 1);
      mbar_init(b_wempty + 8 * i, 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_accfull + 8 * i, 1);
      mbar_init(b_accempty + 8 * i, NUM_EPI_WARPS);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_cready, (uint32_t)(p.csk > 0 ? p.csk * NUM_EPI_WARPS : 1));
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  // Let the next kernel in the stream be scheduled (its CTAs land as SMs free up).
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Cluster split-K: every CTA's barriers are initialised before a peer arrives on them.
  const bool csk = ATMEM && !SWIGLU && p.csk > 0;
  if (csk) cluster_sync_all();

  // This CTA's units: a range of the K steps laid out tile after tile, or, with
  // cluster split-K, its share of one tile's K steps (rank r of s: [r*KS/s, (r+1)*KS/s)).
  long long u_begin, u_end;
  if (csk) {
    const long long tile = blockIdx.x / p.csk, rank = blockIdx.x % p.csk;
    u_begin = tile * p.KS + rank * p.KS / p.csk;
    u_end = tile * p.KS + (rank + 1) * p.KS / p.csk;
  } else {
    u_begin = range_start(p, blockIdx.x);
    u_end = range_start(p, (long long)blockIdx.x + 1);
  }

  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(&g_gemm_error, ERR_TIMEOUT);
  };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return mbar_wait_bounded(bar, parity, abort_flag, WAIT_LIMIT_NS);
  };

  if (warp == 0) {
    // ----------------------------------------------------------- TMA producers --
    // Lane 0 streams the X tiles, lane 1 the raw weight blocks: each runs ahead
    // as far as its own ring allows (W up to SW blocks = 4*SW K steps ahead of
    // the dequantisers, X up to SX steps ahead of the MMA), so a W copy is not
    // held back by the X ring.
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      Ring<XS> rx;
      long long nx = 0;
      bool ok = true;
      UnitIter it{u_begin, u_end, p.KS};
      while (ok && it.next()) {
        const int m0 = locate(p, it.tile).m0;
        for (int k = it.k0; k < it.k1 && ok; ++k) {
#pragma unroll
          for (int t = 0; t < C::XH; ++t) {  // the slots (token halves) of the step
            if (!wait(b_xempty + 8 * rx.s, rx.ph ^ 1u)) {
              ok = false;
              break;
            }
            if (nx == 0) pdl_wait();  // X may come from the previous kernel; the weights do not
#ifdef JLLM_FAULT_INJECTION
            if (!(nx == 0 && blockIdx.x == 0 && g_fi_skip_x))
#endif
            {
              mbar_arrive_expect_tx(b_xfull + 8 * rx.s, x_slot_bytes);
              // one box of 64 k (the 128-byte swizzle atom) x HB tokens per K half
#pragma unroll
              for (int h = 0; h < C::KST / KSTEP; ++h)
                tma_load_2d(sx + (uint32_t)rx.s * x_slot_bytes + (uint32_t)(h * p.HB * KSTEP * 2), &tmX,
                            b_xfull + 8 * rx.s, k * C::KST + h * KSTEP, m0 + t * p.HB);
            }
            rx.next();
            ++nx;
          }
        }
      }
      if (!ok) fail();
      // Every copy this thread issued must have landed before the CTA exits.
      for (long long i = nx > XS ? nx - XS : 0; i < nx; ++i)
        mbar_wait_bounded(b_xfull + 8 * (int)(i % XS), (uint32_t)((i / XS) & 1), nullptr, WAIT_LIMIT_NS);
    } else if (lane == 1) {
      for (int i = 0; i < (SWIGLU ? 2 : p.count); ++i) tma_prefetch_desc(&tmW.w[i]);
      Ring<SW> rw;
      long long nw = 0;
      bool ok = true;
      UnitIter it{u_begin, u_end, p.KS};
      while (ok && it.next()) {
        const TileLoc loc = locate(p, it.tile);
        const CUtensorMap* mw = &tmW.w[loc.b];
        for (int k = it.k0; k < it.k1; ++k) {
          if (k == it.k0 || (k & (C::SPB - 1)) == 0) {
            if (!wait(b_wempty + 8 * rw.s, rw.ph ^ 1u)) {
              ok = false;
              break;
            }
            const uint32_t bar = b_wfull + 8 * rw.s;
            mbar_arrive_expect_tx(bar, W_STAGE_BYTES * NMAT);
            if (SWIGLU) {
              // SwiGLU pairs: tile rows 32g..32g+15 are gate rows n0+16g.., rows
              // 32g+16..32g+31 the up rows of the same outputs (16-row boxes), so that
              // each TMEM lane quarter holds 16 (gate, up) row pairs, lane l and l+16.
              const uint32_t dst = sw + (uint32_t)rw.s * W_STAGE_BYTES;
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                tma_load_3d(dst + (uint32_t)(32 * g) * BLOCK_BYTES, &tmW.w[0], bar, 0, k / C::SPB, loc.n0 + 16 * g);
                tma_load_3d(dst + (uint32_t)(32 * g + 16) * BLOCK_BYTES, &tmW.w[1], bar, 0, k / C::SPB, loc.n0 + 16 * g);
              }
            } else {
              tma_load_3d(sw + (uint32_t)(rw.s * NMAT) * W_STAGE_BYTES, mw, bar, 0, k / C::SPB, loc.n0);
            }
            rw.next();
            ++nw;
          }
        }
      }
      if (!ok) fail();
      for (long long i = nw > SW ? nw - SW : 0; i < nw; ++i)
        mbar_wait_bounded(b_wfull + 8 * (int)(i % SW), (uint32_t)((i / SW) & 1), nullptr, WAIT_LIMIT_NS);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer --
      // Descriptors are a per-stage base plus 2 per K = 16 slice (32 bytes >> 4
      // in the start-address field, which cannot carry within shared memory),
      // and the barriers of step k+1 are probed (non-blocking test) before step
      // k's MMAs are issued so that the probe's latency overlaps the issue.
      const uint32_t idesc = umma_idesc_f16(TILE_N, p.HB);
      const uint64_t adesc0 = umma_desc_sw128(sa), bdesc0 = umma_desc_sw128(sx);
      const uint32_t a_step = (uint32_t)(NMAT * A_STAGE_BYTES) >> 4, b_step = x_slot_bytes >> 4;
      Ring<SA> ra;
      Ring<XS> rx;
      Ring<C::NACC> racc;
      bool ok = true;
      UnitIter it{u_begin, u_end, p.KS};
      while (ok && it.next()) {
        // (wide tiles: this is half 0; half 1 is awaited before its first MMA)
        if (!wait(b_accempty + 8 * racc.s, racc.ph ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)racc.s * C::ACC;
        bool x_ready = mbar_test_wait(b_xfull + 8 * rx.s, rx.ph);
        bool a_ready = C::COMB || mbar_test_wait(b_afull + 8 * ra.s, ra.ph);
        for (int k = it.k0; k < it.k1; ++k) {
          if constexpr (WIDE) {
            // The A stage, then each token half's X slot in turn: a half's four
            // MMAs go out when its box has landed, and its slot is released
            // (commit) as soon as they are done; the A stage after both.
            if (!wait(b_afull + 8 * ra.s, ra.ph)) {
              ok = false;
              break;
            }
            const uint64_t ad = adesc0 + (uint64_t)(ra.s * a_step);
            const uint32_t sa_now = ra.s;
            ra.next();
            const uint32_t acc0 = k > it.k0 ? 1u : 0u;
#pragma unroll
            for (int t = 0; t < C::XH; ++t) {
              if (!wait(b_xfull + 8 * rx.s, rx.ph) || (t == 1 && k == it.k0 && !wait(b_accempty + 8, racc.ph ^ 1u))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t bt = bdesc0 + (uint64_t)(rx.s * b_step);
              const uint32_t dt = d + 256u * t;
#pragma unroll
              for (int kk = 0; kk < KSTEP / 16; ++kk) umma_f16(dt, ad + 2 * kk, bt + 2 * kk, idesc, kk ? 1u : acc0);
              umma_commit(b_xempty + 8 * rx.s);
              rx.next();
            }
            if (!ok) break;
            umma_commit(b_aempty + 8 * sa_now);
            continue;
          }
          if ((!x_ready && !wait(b_xfull + 8 * rx.s, rx.ph)) || (!a_ready && !wait(b_afull + 8 * ra.s, ra.ph))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + (uint64_t)(ra.s * a_step), bd = bdesc0 + (uint64_t)(rx.s * b_step);
          const uint32_t sa_now = ra.s, sx_now = rx.s;
          ra.next();
          rx.next();
          if (k + 1 < it.k1) {
            x_ready = mbar_test_wait(b_xfull + 8 * rx.s, rx.ph);
            a_ready = C::COMB || mbar_test_wait(b_afull + 8 * ra.s, ra.ph);
          }
          const uint32_t acc0 = k > it.k0 ? 1u : 0u;
          if (ATMEM) {
            const uint32_t at = tmem + A_TMEM_COL0 + sa_now * C::ASC;
            const uint32_t half = (uint32_t)(p.BN * KSTEP * 2) >> 4;  // second 64-wide X box of the step
#pragma unroll
            for (int kk = 0; kk < C::KST / 16; ++kk)
              umma_f16_ta(d, at + 8 * kk, bd + (kk >> 2) * half + 2 * (kk & 3), idesc, kk ? 1u : acc0);
          } else {
            umma_f16(d, ad, bd, idesc, acc0);
#pragma unroll
            for (int kk = 1; kk < KSTEP / 16; ++kk) umma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, 1u);
          }
          if (!C::COMB) umma_commit(b_aempty + 8 * sa_now);
          umma_commit(b_xempty + 8 * sx_now);
        }
        if (!ok) break;
        umma_commit(b_accfull + 8 * racc.s);
        racc.next();
      }
      if (!ok) fail();
      umma_commit(b_drain);  // tracks every MMA issued, also after an abort
      mbar_wait_bounded(b_drain, 0, nullptr, WAIT_LIMIT_NS);
    }
  } else if (warp < EPI_WARP0) {
    // --------------------------------------------------------------- dequant --
    // Warp w handles TMEM lane quarter q = w & 3 (rows 32q..32q+31) and half
    // hw = (w - 2) >> 2 of each step.  64-wide steps: hw is the nibble side --
    // hw = 0 makes sub-block 2c (low nibbles, k 0..31 of the step), hw = 1
    // sub-block 2c+1 (high nibbles, k 32..63).  128-wide steps: hw is the
    // 64-weight chunk of the step, and the warp makes both of its sub-blocks.
    const int q = warp & 3;
    const int hw = (warp - 2) >> 2;
    const int r = 32 * q + lane;
    constexpr int NH = C::KST / KSTEP;  // sub-block halves per thread and step
    Ring<SA> ra;
    Ring<SW> rw;
    bool ok = true;
    UnitIter it{u_begin, u_end, p.KS};
    while (ok && it.next()) {
      for (int k = it.k0; k < it.k1; ++k) {
        const int ks = k & (C::SPB - 1);  // step within the super-block
        const int c = NH == 2 ? 2 * ks + hw : ks;  // this thread's 64-weight chunk of the block
        // Waits are made warp-uniform so that a timeout leaves the warp converged.
        if (k == it.k0 || ks == 0) ok = __all_sync(0xffffffffu, wait(b_wfull + 8 * rw.s, rw.ph));
        if (ok) ok = __all_sync(0xffffffffu, wait((C::COMB ? b_xempty : b_aempty) + 8 * ra.s, ra.ph ^ 1u));
        if (!ok) break;
#pragma unroll
        for (int mat = 0; mat < NMAT; ++mat) {
          const uint8_t* raw = smem + p.off_w + (size_t)(rw.s * NMAT + mat) * W_STAGE_BYTES + (size_t)r * BLOCK_BYTES;
          const uint4 hd = *reinterpret_cast<const uint4*>(raw);
          const uint4 q0 = *reinterpret_cast<const uint4*>(raw + 16 + 32 * c);
          const uint4 q1 = *reinterpret_cast<const uint4*>(raw + 32 + 32 * c);
          const unsigned short d16 = (unsigned short)(hd.x & 0xffffu);
          const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int hi = 0; hi < NH; ++hi) {
            const int hs = NH == 2 ? hi : hw;  // nibble side: sub-block 2c + hs
            uint32_t sc, m;
            q4k_scale_min(hd.y, hd.z, hd.w, 2 * c + hs, sc, m);
            // p = sc*q exactly in fp16 from the offset code h (1024+q or 1024+16q):
            //   p = h*sc - 1024*sc  or  p = h*(sc/16) - 64*sc   (one rounding of an
            //   exact integer <= 945).  Then w = fma(d, p, -dmin*m) in fp32 is the
            //   exact value rounded once, i.e. the fp32 dequant, rounded to fp16.
            const uint32_t mask = hs ? 0x00F000F0u : 0x000F000Fu;
            const __half sch = __uint2half_rn(sc);
            const __half2 scv = __half2half2(hs ? __hmul(sch, __float2half(0.0625f)) : sch);
            const __half2 offv = __half2half2(__hmul(sch, __float2half(hs ? -64.f : -1024.f)));
            const uint32_t scv_u = *reinterpret_cast<const uint32_t*>(&scv);
            const uint32_t offv_u = *reinterpret_cast<const uint32_t*>(&offv);
            const float nt = -__fmul_rn(half_hi_to_float(hd.x), (float)m);
            uint32_t pk[16];  // fp16 pairs (k, k+1) for k = 32*hs + 2*i of the chunk
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t wp;
              asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(wp) : "r"(qw[i]));  // bytes b0 b2 b1 b3
              pk[2 * i] = dq_pair(lop3_and_or(wp, mask, 0x64006400u), scv_u, offv_u, d16, nt);           // k, k+1
              pk[2 * i + 1] = dq_pair(lop3_and_or(wp >> 8, mask, 0x64006400u), scv_u, offv_u, d16, nt);  // k+2, k+3
            }
            if (ATMEM) {
              // lane r of the warp's TMEM quarter, 16 columns of the stage (two fp16 per column):
              // the chunk's 32 columns at 32*hw (128-wide steps), the sub-block's half at 16*hs
              tmem_st16(tmem + ((uint32_t)(32 * q) << 16) + A_TMEM_COL0 + ra.s * C::ASC + (NH == 2 ? 32 * hw : 0) +
                            16 * hs,
                        pk);
            } else {
              uint8_t* arow = smem + p.off_a + (size_t)(ra.s * NMAT + mat) * A_STAGE_BYTES + (size_t)r * 128;
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {  // output chunk j8 = 4*hs + jj holds k = 8*j8..8*j8+7
                const int j8 = 4 * hs + jj;
                *reinterpret_cast<uint4*>(arow + ((j8 ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]);
              }
            }
          }
        }
        if (ATMEM) tc_fence_before();
        else fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive((C::COMB ? b_xfull : b_afull) + 8 * ra.s);
        ra.next();
        if (k == it.k1 - 1 || ks == C::SPB - 1) {
          if (lane == 0) mbar_arrive(b_wempty + 8 * rw.s);
          rw.next();
        }
      }
    }
    if (!ok && lane == 0) fail();
  } else {
    // -------------------------------------------------------------- epilogue --
    // Warp w reads TMEM lane quarter q = w & 3: rows 32q..32q+31 of the tile.
    const int q = warp & 3;
    const int r = 32 * q + lane;
    pdl_wait();  // Y, the partial slots and the flags are touched only after the previous kernel
    Ring<C::NACC> racc;
    // TMEM column of the tile's token column cc (a multiple of 32): wide tiles
    // keep their second token half at column 256.
    auto tcol = [&](int cc) -> uint32_t { return (uint32_t)(WIDE && cc >= p.HB ? 256 + cc - p.HB : cc); };
    // This warp is done reading accumulator buffer (wide tiles: half) i.
    auto release = [&](int i) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_accempty + 8 * i);
    };
    bool ok = true;
    UnitIter it{u_begin, u_end, p.KS};
    while (ok && it.next()) {
      ok = mbar_wait_warp_sleepy(b_accfull + 8 * racc.s, racc.ph, abort_flag, WAIT_LIMIT_NS);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)racc.s * C::ACC;
      const TileLoc loc = locate(p, it.tile);
      const int n = loc.n0 + r, m0 = loc.m0;
      const bool writer = !csk && it.k0 > 0;          // later part of a cut tile
      const bool fixer = !csk && !writer && it.k1 < p.KS;  // first part of a cut tile
      if (csk) {
        // Cluster split-K (the CTA's one unit): its fp32 partial of the tile goes
        // to its own X ring ([column][row]; the ring is idle once the unit's MMAs
        // are done), every CTA of the cluster is told that this warp's rows are in
        // place, and then this CTA adds up its slice of the tile's rows -- the
        // cluster's partials in rank (= K) order, read through distributed shared
        // memory -- and stores that slice of Y.
        float* part = reinterpret_cast<float*>(smem + p.off_x);
        for (int cc = 0; cc < p.BN; cc += 32) {
          uint32_t v[32];
          tmem_ld32(tl + cc, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) part[(size_t)(cc + j) * TILE_N + r] = __uint_as_float(v[j]);
        }
        release(racc.s);  // (its __syncwarp orders the lanes' stores before lane 0's release-arrivals)
        if (lane == 0)
          for (int d = 0; d < p.csk; ++d) mbar_arrive_remote(mapa_shared(b_cready, (uint32_t)d));
        int rok = 1;
        if (lane == 0) rok = mbar_wait_cluster_bounded(b_cready, 0, WAIT_LIMIT_NS) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, rok, 0) != 0;
        __syncwarp();
        if (!ok) break;
        // This CTA's slice: 4-row groups [rank*32/s, (rank+1)*32/s) of all BN
        // columns; a thread takes one (column, 4-row group) at a time, with
        // every peer's 16 bytes loaded before the adds.
        const int rank = (int)(blockIdx.x % (unsigned)p.csk);
        const int g0 = rank * (TILE_N / 4) / p.csk, ng = (rank + 1) * (TILE_N / 4) / p.csk - g0;
        const uint32_t part_u32 = smem_u32(part);
        const int tid = (int)threadIdx.x - EPI_WARP0 * 32;  // 0..127
        const bool vec = (loc.N & 3) == 0;                  // whole 4-row groups of Y are 16 / 8 bytes aligned
        auto store4 = [&](int col, int row, float4 a) {
          const int nn = loc.n0 + row, m = m0 + col;
          if (m >= p.M) return;
          const size_t o = (size_t)m * loc.N + nn;
          if (vec && nn + 3 < loc.N) {
            if (p.out_f16) {
              const __half2 lo = __floats2half2_rn(a.x, a.y), hi = __floats2half2_rn(a.z, a.w);
              *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(loc.y) + o) =
                  make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
            } else {
              *reinterpret_cast<float4*>(reinterpret_cast<float*>(loc.y) + o) = a;
            }
          } else {
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (nn + i < loc.N) {
                if (p.out_f16) reinterpret_cast<__half*>(loc.y)[o + i] = __float2half_rn(av[i]);
                else reinterpret_cast<float*>(loc.y)[o + i] = av[i];
              }
          }
        };
        const int items = ng * p.BN;
        for (int e = tid; e < items; e += NUM_EPI_WARPS * 32) {
          const int row = 4 * (g0 + e % ng), col = e / ng;  // consecutive threads: consecutive row groups
          const uint32_t off = (uint32_t)((col * TILE_N + row) * 4);
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int d0 = 0; d0 < p.csk; d0 += 4) {  // four peers' loads in flight, added in rank order
            float4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              v[i] = ld_cluster_f32x4(mapa_shared(part_u32 + off, (uint32_t)(d0 + i < p.csk ? d0 + i : d0)));
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (d0 + i < p.csk) a.x += v[i].x, a.y += v[i].y, a.z += v[i].z, a.w += v[i].w;
          }
          store4(col, row, a);
        }
      } else if (writer) {
        // Leave the fp32 partial in this CTA's slot, then count this warp in
        // the slot's flag.  Slot layout [column / 4][row][column % 4]: a warp
        // moves 16 bytes per row, 512 contiguous bytes per access.
        float4* slot = reinterpret_cast<float4*>(p.partial + (size_t)blockIdx.x * SLOT_FLOATS) + r;
        {
          for (int cc = 0; cc < p.BN; cc += 32) {
            uint32_t v[32];
            tmem_ld32(tl + tcol(cc), v);
            if (WIDE && cc + 32 == p.HB) release(0);  // half 0 is in registers
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcg(slot + (size_t)(cc / 4 + i) * TILE_N,
                     make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
          }
        }
        release(WIDE ? 1 : racc.s);
        __threadfence();
        __syncwarp();
        if (lane == 0) atom_add_release_gpu(p.flags + blockIdx.x, 1u);
      } else {
        // Contributors to a cut tile: the CTAs after this one whose ranges
        // start inside it, summed in CTA order.
        int j_end = blockIdx.x + 1;
        if (fixer) {
          const long long tile_end = (long long)(it.tile + 1) * p.KS;
          while (j_end < (int)gridDim.x && range_start(p, j_end) < tile_end) ++j_end;
          for (int j = blockIdx.x + 1; j < j_end && ok; ++j) {
            bool ready = false;
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t it2 = 0;; ++it2) {
              if (ld_acquire_gpu(p.flags + j) >= (uint32_t)NUM_EPI_WARPS) {
                ready = true;
                break;
              }
              if ((it2 & 63u) == 63u && (*abort_flag || globaltimer_ns() - t0 > WAIT_LIMIT_NS)) break;
            }
            ok = __all_sync(0xffffffffu, ready);
          }
          if (!ok) break;
        }
        // The contributors' partial sums, added in CTA order.  Wide tiles: the
        // sums of chunk cc + 32 are loaded before chunk cc's stores, so that
        // their latency overlaps the stores and the next tensor-memory read
        // (the other variants have no registers to spare for it).
        const bool summed = j_end > (int)blockIdx.x + 1;
        const float4* slot0 = reinterpret_cast<const float4*>(p.partial + (size_t)(blockIdx.x + 1) * SLOT_FLOATS) + r;
        constexpr size_t SLOT4 = SLOT_FLOATS / 4;
        constexpr bool PIPE = WIDE;
        float4 nx[8];
        if (PIPE && summed) {
#pragma unroll
          for (int i = 0; i < 8; ++i) nx[i] = __ldcg(slot0 + (size_t)i * TILE_N);
          for (int jc = blockIdx.x + 2; jc < j_end; ++jc)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 t = __ldcg(slot0 + (size_t)(jc - blockIdx.x - 1) * SLOT4 + (size_t)i * TILE_N);
              nx[i].x += t.x, nx[i].y += t.y, nx[i].z += t.z, nx[i].w += t.w;
            }
        }
        for (int cc = 0; cc < p.BN; cc += 32) {
          uint32_t v[32];
          tmem_ld32(tl + tcol(cc), v);
          if (WIDE && cc + 32 == p.HB) release(0);  // half 0 is in registers
          float a[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = __uint_as_float(v[j]);
          if (!PIPE) {
            for (int jc = blockIdx.x + 1; jc < j_end; ++jc) {
              const float4* slot = reinterpret_cast<const float4*>(p.partial + (size_t)jc * SLOT_FLOATS) +
                                   (size_t)(cc / 4) * TILE_N + r;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 t = __ldcg(slot + (size_t)i * TILE_N);
                a[4 * i] += t.x, a[4 * i + 1] += t.y, a[4 * i + 2] += t.z, a[4 * i + 3] += t.w;
              }
            }
          } else if (summed) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              a[4 * i] += nx[i].x, a[4 * i + 1] += nx[i].y, a[4 * i + 2] += nx[i].z, a[4 * i + 3] += nx[i].w;
            if (cc + 32 < p.BN) {
              const float4* slot = slot0 + (size_t)((cc + 32) / 4) * TILE_N;
#pragma unroll
              for (int i = 0; i < 8; ++i) nx[i] = __ldcg(slot + (size_t)i * TILE_N);
              for (int jc = blockIdx.x + 2; jc < j_end; ++jc)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 t = __ldcg(slot + (size_t)(jc - blockIdx.x - 1) * SLOT4 + (size_t)i * TILE_N);
                  nx[i].x += t.x, nx[i].y += t.y, nx[i].z += t.z, nx[i].w += t.w;
                }
            }
          }
          const int jv = min(32, min(p.BN - cc, p.M - (m0 + cc)));
          if (SWIGLU) {
            // Lane l < 16 holds gate row n0+16q+l, lane l+16 the up row of the same
            // output.  The gate lane makes h for tokens 0..15 of the chunk, the up
            // lane for 16..31: each sends the partner the value of the partner's
            // token (one exchange per token) and keeps its own.  The 16 exchanges go
            // first, so that the silu chains of different tokens overlap.
            const int no = loc.n0 + 16 * q + (lane & 15);
            const bool up_lane = lane >= 16;
            __half* yp = reinterpret_cast<__half*>(loc.y) + (size_t)(m0 + cc + (up_lane ? 16 : 0)) * loc.N + no;
            const int jmax = jv - (up_lane ? 16 : 0);
            float o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = __shfl_xor_sync(0xffffffffu, up_lane ? a[j] : a[j + 16], 16);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float mine = up_lane ? a[j + 16] : a[j];
              const float g = up_lane ? o[j] : mine, u = up_lane ? mine : o[j];
              if (j < jmax && no < loc.N) yp[(size_t)j * loc.N] = __float2half_rn(__fdividef(g, 1.0f + __expf(-g)) * u);
            }
          } else if (n < loc.N && jv > 0) {
            // Y[m0+cc+j][n] for the j in range: one pointer step of N per token, the
            // bounds tested once per chunk.
            const size_t off = (size_t)(m0 + cc) * loc.N + n;
            const size_t ld = (size_t)loc.N;
            if (p.out_f16) {
              __half* yp = reinterpret_cast<__half*>(loc.y) + off;
              if (jv == 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j) yp[j * ld] = __float2half_rn(a[j]);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j < jv) yp[j * ld] = __float2half_rn(a[j]);
              }
            } else {
              float* yp = reinterpret_cast<float*>(loc.y) + off;
              if (jv == 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j) yp[j * ld] = a[j];
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j < jv) yp[j * ld] = a[j];
              }
            }
          }
        }
        release(WIDE ? 1 : racc.s);
        if (lane == 0) {
          // The last of the four epilogue warps to finish returns the
          // contributors' flags to zero for the next call.
          for (int jc = blockIdx.x + 1; jc < j_end; ++jc)
            if (atom_add_acqrel_gpu(p.flags + jc, 1u) == 2 * NUM_EPI_WARPS - 1) p.flags[jc] = 0;
        }
      }
      racc.next();
    }
    if (!ok && lane == 0) fail();
  }

  tc_fence_before();
  __syncthreads();
  // Cluster split-K: no CTA leaves while its peers may still read its partial.
  if (csk) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
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

// Encoded tensor maps depend only on the device, the base address, the extents
// and the box, so repeated calls on the same buffers reuse them: a small table
// with least-recently-used replacement, shared by all threads under a mutex.
struct MapKey {
  int dev, kind;  // kind 0: X map, 1: W map
  const void* ptr;
  int64_t a, b;   // X: M, K; W: N, K
  int box;        // X: tokens per tile; W: 0
  bool operator==(const MapKey& o) const {
    return dev == o.dev && kind == o.kind && ptr == o.ptr && a == o.a && b == o.b && box == o.box;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  uint64_t stamp = 0;  // 0: empty
};
constexpr int kMapCache = 64;
MapEntry g_map_cache[kMapCache];
uint64_t g_map_clock = 0;
std::mutex g_map_mu;

bool map_lookup(const MapKey& k, CUtensorMap* out) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (MapEntry& e : g_map_cache)
    if (e.stamp && e.key == k) {
      e.stamp = ++g_map_clock;
      *out = e.map;
      return true;
    }
  return false;
}

void map_insert(const MapKey& k, const CUtensorMap& m) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry* victim = &g_map_cache[0];
  for (MapEntry& e : g_map_cache) {
    if (e.stamp == 0) {
      victim = &e;
      break;
    }
    if (e.stamp < victim->stamp) victim = &e;
  }
  victim->key = k;
  victim->map = m;
  victim->stamp = ++g_map_clock;
}

cudaError_t make_x_map(const void* x, int64_t M, int64_t K, int BN, CUtensorMap* mx) {
  const MapKey key{device_info().device, 0, x, M, K, BN};
  if (map_lookup(key, mx)) return cudaSuccess;
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {KSTEP, (cuuint32_t)BN};
  const cuuint32_t es[2] = {1, 1};
  if (enc(mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  map_insert(key, *mx);
  return cudaSuccess;
}

// Byte view of a packed weight matrix: (144 bytes, super-block, row), one
// super-block of box_rows rows per load (128, or 16 for the SwiGLU pairs).
cudaError_t make_w_map(const void* w, int64_t N, int64_t K, CUtensorMap* mw, int box_rows = TILE_N) {
  const MapKey key{device_info().device, 1, w, N, K, box_rows};
  if (map_lookup(key, mw)) return cudaSuccess;
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  const int64_t NB = K / QK;
  const cuuint64_t wdims[3] = {(cuuint64_t)BLOCK_BYTES, (cuuint64_t)NB, (cuuint64_t)N};
  const cuuint64_t wstrides[2] = {(cuuint64_t)BLOCK_BYTES, (cuuint64_t)(NB * BLOCK_BYTES)};
  const cuuint32_t wbox[3] = {BLOCK_BYTES, 1, (cuuint32_t)box_rows};
  const cuuint32_t wes[3] = {1, 1, 1};
  if (enc(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w), wdims, wstrides, wbox, wes,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  map_insert(key, *mw);
  return cudaSuccess;
}

// Launch-shape constants of the GEMM:
//   bn     tokens per tile (0: chosen per launch; else a multiple of 16 up to
//          the kernel's cap)
//   split  0 keeps whole tiles even when a workspace is given
// They are fixed in the shipped library.  A build with -DJLLM_TUNING reads
// overrides once from the environment (JLLM_GEMM_BN, JLLM_GEMM_SPLIT), for
// measurements only.
//   atmem  1: the A operand in tensor memory (single-GEMM and batched launches)
//   wide   1: tiles of up to 512 tokens when M > 256 and they fill the SMs
//          (single-GEMM and batched); 2: whenever M > 256
//   csk    1: cluster split-K for narrow tiles that do not fill the SMs
struct GemmKnobs {
  int bn = 0;
  int split = 1;
  int atmem = 1;
  int wide = 1;
  int csk = 1;
};
const GemmKnobs& gemm_knobs() {
  static GemmKnobs k = [] {
    GemmKnobs v;
#ifdef JLLM_TUNING
    if (const char* e = getenv("JLLM_GEMM_BN")) v.bn = atoi(e);
    if (const char* e = getenv("JLLM_GEMM_SPLIT")) v.split = atoi(e);
    if (const char* e = getenv("JLLM_GEMM_ATMEM")) v.atmem = atoi(e);
    if (const char* e = getenv("JLLM_GEMM_WIDE")) v.wide = atoi(e);
    if (const char* e = getenv("JLLM_GEMM_CSK")) v.csk = atoi(e);
#endif
    return v;
  }();
  return k;
}

// Clusters of `cs` CTAs of the narrow-tile kernel (cluster split-K) that can be
// resident at once with `smem` bytes of shared memory each; cached per
// (device, cluster size, shared memory).
int max_active_clusters(int cs, size_t smem) {
  struct Entry {
    int dev, cs;
    size_t smem;
    int n;
  };
  static Entry cache[32];
  static int used = 0;
  static std::mutex mu;
  const int dev = device_info().device;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].cs == cs && cache[i].smem == smem) return cache[i].n;
  auto kern = q4k_gemm_tc_kernel<false, true, false>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
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
  if (used < 32) cache[used++] = Entry{dev, cs, smem, n};
  return n;
}

template <bool SWIGLU, bool ATMEM, bool WIDE = false>
cudaError_t launch_tc(const CUtensorMap& mx, const WMaps& mw, const GemmParams& p, int grid, bool cooperative,
                      size_t smem, cudaStream_t s, int cluster = 0) {
  auto kern = q4k_gemm_tc_kernel<SWIGLU, ATMEM, WIDE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  unsigned n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
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

// Library-owned workspace of jllm_q4k_gemm_noalloc: zero at module load,
// returned to zero by every call that completes.  Sized for up to
// kStaticWsSMs SMs.
constexpr int kStaticWsSMs = 160;
constexpr size_t kStaticWsBytes =
    ((size_t)kStaticWsSMs * SLOT_FLOATS * sizeof(float) + (size_t)kStaticWsSMs * sizeof(uint32_t) + 255) & ~(size_t)255;
__device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
void* g_static_ws_ptr[kMaxDevices];
cudaError_t g_static_ws_err[kMaxDevices];
std::once_flag g_static_ws_once[kMaxDevices];
std::atomic<bool> g_static_ws_ready[kMaxDevices];

}  // namespace

cudaError_t gemm_static_workspace(void** ptr, size_t* bytes) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_static_ws_once[d], [d]() {
    g_static_ws_err[d] = cudaGetSymbolAddress(&g_static_ws_ptr[d], g_static_ws);
    if (g_static_ws_err[d] == cudaSuccess) g_static_ws_ready[d].store(true);
  });
  if (g_static_ws_err[d] != cudaSuccess) return g_static_ws_err[d];
  *ptr = g_static_ws_ptr[d];
  *bytes = kStaticWsBytes;
  return cudaSuccess;
}

// After a kernel-side timeout the stream-K flag words of the static workspace
// can be left non-zero (a contributor counted in, its finishing CTA gave up);
// a later call would take them for fresh partial sums.  Return them to zero
// (the partial slots need no clearing: a contributor rewrites its slot before
// it counts in).  Nothing to do on a device whose array was never used.
cudaError_t gemm_static_workspace_reset(cudaStream_t s) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= kMaxDevices || !g_static_ws_ready[d].load()) return cudaSuccess;
  const DevInfo& dev = device_info();
  if (dev.err != cudaSuccess) return dev.err;
  const size_t off = (size_t)dev.sm_count * SLOT_FLOATS * sizeof(float);
  e = cudaMemsetAsync(static_cast<uint8_t*>(g_static_ws_ptr[d]) + off, 0, (size_t)dev.sm_count * sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

size_t gemm_workspace_bytes() {
  const DevInfo& dev = device_info();
  if (dev.err != cudaSuccess || dev.sm_count <= 0) return 0;
  const size_t bytes = (size_t)dev.sm_count * SLOT_FLOATS * sizeof(float) + (size_t)dev.sm_count * sizeof(uint32_t);
  return (bytes + 255) & ~(size_t)255;
}

namespace {

// One launch over `count` weight matrices sharing X (count 1 with w1 set:
// SwiGLU of gate w[0] and up w1 into one fp16 output).
cudaError_t launch_tc_common(const void* const* w, const void* w1, const int64_t* Ns, int count, const void* x,
                             void* const* y, bool y_f16, int64_t M, int64_t K, void* ws, size_t ws_bytes,
                             cudaStream_t s) {
  const DevInfo& dev = device_info();
  // SwiGLU (w1 = up): one matrix of tiles whose 128 rows pair 64 gate and 64 up
  // rows (the kernel's pair mode), so it takes the plain tile shapes.
  const bool swiglu = w1 != nullptr;
  const int nmat = 1;
  const int64_t rows_per_tile = swiglu ? TILE_N / 2 : TILE_N;  // output columns per tile
  if (count < 1 || count > kBatchMax || (swiglu && count != 1)) return cudaErrorInvalidValue;
  if (M > INT32_MAX / 2 || K / QK > INT32_MAX / 8) return cudaErrorInvalidValue;
  const GemmKnobs& kn = gemm_knobs();
  // Tokens per tile: the whole of M up to the cap (rounded up to 16), else
  // the cap (256).
  int bn_cap = Cfg<false>::BN_MAX;
  if (kn.bn >= 16 && kn.bn <= bn_cap && kn.bn % 16 == 0) bn_cap = kn.bn;
  int BN = (int)((M + 15) / 16 * 16);
  if (BN > bn_cap) BN = bn_cap;
  // A mid-size M (one token tile, more than half the cap) over few weight-row
  // tiles: two token tiles of half the size put twice the CTAs to work while
  // they still fit in one wave (each weight tile is then dequantised twice).
  int64_t n_tiles = 0;
  for (int b = 0; b < count; ++b) n_tiles += Ns[b] > 0 ? (Ns[b] + rows_per_tile - 1) / rows_per_tile : 0;
  if (kn.bn == 0 && M > bn_cap / 2 && M <= bn_cap && 2 * n_tiles <= dev.sm_count)
    BN = (int)(((M + 1) / 2 + 15) / 16 * 16);
  // Tiles of at most 128 tokens keep the dequantised A operand in tensor memory
  // (9-12 % faster than in shared memory at the same tile width, measured at 128
  // and 192 tokens), with 128-wide K steps; wider tiles need all 512 columns for
  // two accumulators.
  const bool atmem = kn.atmem != 0 && BN <= Cfg<false, true>::BN_MAX;
  // More than 256 tokens: wide tiles of up to 512 (the fewest tiles of at most
  // 512 tokens, each a multiple of 64, so that the halves are multiples of 32),
  // when there are at least as many as SMs.  Fewer would leave SMs idle or be
  // cut between CTAs, and a cut wide tile's fix-up (256 KiB of partial sums per
  // contributor) costs more than the wide tile saves.
  using CW = Cfg<false, false, true>;
  bool wide = false;
  // (Not for SwiGLU: its epilogue -- an exchange and a silu per output -- is
  // slow enough that the single accumulator of a wide tile would wait for it;
  // two 256-token accumulators hide it: 189.8 against 221.9 us for gate/up
  // 2560 -> 2 x 9728 at M = 2048.)
  if (!swiglu && kn.wide != 0 && kn.bn == 0 && M > 256) {
    const int64_t mt = (M + CW::BN_MAX - 1) / CW::BN_MAX;
    if (mt * n_tiles >= (kn.wide > 1 ? 1 : dev.sm_count)) {
      wide = true;
      BN = (int)(((M + mt - 1) / mt + 63) / 64 * 64);
    }
  }
  const int HB = wide ? BN / 2 : BN;

  GemmParams p = {};
  p.M = (int)M;
  p.NB = (int)(K / QK);
  p.BN = BN;
  p.HB = HB;
  p.m_tiles = (int)((M + BN - 1) / BN);
  const int kst = atmem ? Cfg<false, true>::KST : KSTEP;  // K per pipeline step
  p.KS = (QK / kst) * p.NB;
  p.out_f16 = (y_f16 || swiglu) ? 1 : 0;
  p.pair = swiglu ? 1 : 0;
  p.count = count;
  long long tiles = 0;
  for (int b = 0; b < count; ++b) {
    if (Ns[b] < 1 || Ns[b] > INT32_MAX / 2) return cudaErrorInvalidValue;
    p.y[b] = y[b];
    p.N[b] = (int)Ns[b];
    p.tile0[b] = (int)tiles;
    tiles += (long long)p.m_tiles * ((Ns[b] + rows_per_tile - 1) / rows_per_tile);
    if (tiles > INT32_MAX / 2) return cudaErrorInvalidValue;
  }
  p.tile0[count] = (int)tiles;
  const long long units = tiles * p.KS;
  if (units > (1ll << 53)) return cudaErrorInvalidValue;
  const int sms = dev.sm_count;

  // Stream-K when the tiles do not fill the SMs evenly and a workspace is
  // given; each CTA then takes at least 8 K steps.  It pays only if it shortens
  // the busiest CTA by more than the cut tiles' fix-up, about 12 K steps
  // (measured at M = 235: q/k/v, 96 tiles of 20 steps, 17.8 us whole against
  // 21.9 split; o, 40 of 32, 24.0 against 22.8; down, 40 of 76, 51.8 against 31.1).
  bool split = kn.split != 0 && ws != nullptr && ws_bytes >= gemm_workspace_bytes() && tiles % sms != 0;
  long long g = units / 8;
  if (g > sms) g = sms;
  if (g < 1) g = 1;
  if (split && ((tiles + sms - 1) / sms) * p.KS - (units + g - 1) / g < 12) split = false;
  int grid;
  if (split) {
    grid = (int)g;
    p.grain = 1;
    p.grains = units;
    p.partial = reinterpret_cast<float*>(ws);
    p.flags = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(ws) + (size_t)sms * SLOT_FLOATS * sizeof(float));
  } else {
    grid = (int)(tiles < sms ? tiles : sms);
    p.grain = p.KS;
    p.grains = tiles;
  }

  // Shared memory: X ring, dequantised-A ring (not with A in tensor memory),
  // raw-W ring, barriers.
  const int SX = atmem ? Cfg<false, true>::SX : (wide ? CW::SX : Cfg<false>::SX);
  const int SA = atmem ? Cfg<false, true>::SA : (wide ? CW::SA : Cfg<false>::SA);
  const int SW = atmem ? Cfg<false, true>::SW : (wide ? CW::SW : Cfg<false>::SW);
  const int nbars = atmem ? Cfg<false, true>::NBARS : (wide ? CW::NBARS : Cfg<false>::NBARS);
  p.x_stage_bytes = (uint32_t)BN * kst * 2;
  p.off_x = 0;
  p.off_a = (uint32_t)SX * p.x_stage_bytes;
  p.off_w = p.off_a + (atmem ? 0u : (uint32_t)(SA * nmat * A_STAGE_BYTES));
  p.off_bar = p.off_w + (uint32_t)(SW * nmat * W_STAGE_BYTES);
  const size_t smem = 1024 + p.off_bar + 8 * nbars + 16;
  if (smem > dev.smem_optin) return cudaErrorInvalidValue;

  // Cluster split-K for narrow tiles that are few next to the SMs: a cluster
  // of s CTAs per tile, each taking 1/s of its K steps, the partials added
  // through distributed shared memory -- no workspace, no flags, no cut-tile
  // tail.  s is the largest of 4..8 (and at most the K steps) for which all
  // the tiles' clusters can be resident at once.  Measured per launch (M = 33
  // to 235): with 7 CTAs per tile (20 tiles) the launch takes 0.67-0.9x the
  // time of the stream-K split, whose cut tiles then have ~7 contributors;
  // with 3 per tile (40-48 tiles) it is 0.94-1.22x, so those keep stream-K.
  int csk = 0;
  if (atmem && !swiglu && kn.csk != 0 && tiles < sms) {  // (a CTA's row slice would split SwiGLU pairs)
    int cs = (int)(sms / tiles);
    if (cs > 8) cs = 8;
    if (cs > p.KS) cs = p.KS;
    for (; cs >= 4; --cs)
      if (max_active_clusters(cs, smem) >= tiles) break;
    if (cs >= 4) csk = cs;
  }
  if (csk) {
    p.csk = csk;
    grid = (int)tiles * csk;
    split = false;
    p.partial = nullptr;
    p.flags = nullptr;
  }

  CUtensorMap mx;
  WMaps mw;
  memset(&mw, 0, sizeof(mw));
  cudaError_t e = make_x_map(x, M, K, HB, &mx);
  for (int b = 0; b < count && e == cudaSuccess; ++b) e = make_w_map(w[b], Ns[b], K, &mw.w[b], swiglu ? 16 : TILE_N);
  if (e == cudaSuccess && swiglu) e = make_w_map(w1, Ns[0], K, &mw.w[1], 16);
  if (e != cudaSuccess) return e;
  if (swiglu)
    return atmem ? launch_tc<true, true>(mx, mw, p, grid, split, smem, s)
                 : launch_tc<true, false>(mx, mw, p, grid, split, smem, s);
  if (wide) return launch_tc<false, false, true>(mx, mw, p, grid, split, smem, s);
  return atmem ? launch_tc<false, true>(mx, mw, p, grid, split, smem, s, csk)
               : launch_tc<false, false>(mx, mw, p, grid, split, smem, s);
}

}  // namespace

cudaError_t launch_gemm_tc(const void* w0, const void* w1, const void* x, void* y, bool y_f16, int64_t M,
                           int64_t N, int64_t K, void* ws, size_t ws_bytes, cudaStream_t s) {
  return launch_tc_common(&w0, w1, &N, 1, x, &y, y_f16, M, K, ws, ws_bytes, s);
}

cudaError_t launch_gemm_tc_batch(const void* const* w, const int64_t* N, int count, const void* x, void* const* y,
                                 bool y_f16, int64_t M, int64_t K, void* ws, size_t ws_bytes, cudaStream_t s) {
  return launch_tc_common(w, nullptr, N, count, x, y, y_f16, M, K, ws, ws_bytes, s);
}

cudaError_t tma_map_x(const void* x, int64_t M, int64_t K, int box_tokens, CUtensorMap* map) {
  return make_x_map(x, M, K, box_tokens, map);
}

cudaError_t tma_map_w(const void* w, int64_t N, int64_t K, int box_rows, CUtensorMap* map) {
  return make_w_map(w, N, K, map, box_rows);
}

#ifdef JLLM_FAULT_INJECTION
cudaError_t fault_injection_set_gemm(int skip_x) { return cudaMemcpyToSymbol(g_fi_skip_x, &skip_x, sizeof(int)); }
#endif

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

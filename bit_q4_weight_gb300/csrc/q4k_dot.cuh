// The one-token Q4_K inner product shared by the GEMV kernels (gemv.cu,
// gemv_chain.cu): one lane's 64-weight chunk of one block row against x.
//
// Each code byte becomes two fp16 values by one AND per pair: the low nibble
// left in place is the fp16 subnormal q*2^-24, the high nibble left at bits
// 4..7 is 16q*2^-24 -- exact, with no offset to remove afterwards.  Their
// products with x are accumulated in fp32 by fma.rn.f32.f16 (exact products);
// per sub-block j, A_j = 2^-24 * sum q_i x_i (16x that for high nibbles), and
// with the staged sums X_j * 2^-24 of x,
//     sum_i w_i x_i = 2^24 * ( d*sc_j * A_j (/16) - dmin*m_j * X_j*2^-24 ),
// the block value d*sc_j*q - dmin*m_j summed against x.  x is staged in
// shared memory as 128-byte chunks (kb, c) of 64 values, 144 bytes apart
// (x_unit_pos), with the 32-element sums X_j.
#pragma once

#include "common.cuh"

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

// acc += lo + hi of an fp16 pair, each added exactly widened (fp16 * 1 + fp32).
__device__ __forceinline__ void add_halves(float& acc, uint32_t h2) {
  asm("{\n .reg .b16 a, b, one;\n mov.b32 {a, b}, %1;\n mov.b16 one, 0x3C00;\n"
      " fma.rn.f32.f16 %0, a, one, %0;\n fma.rn.f32.f16 %0, b, one, %0;\n}"
      : "+f"(acc)
      : "r"(h2));
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

__device__ __forceinline__ uint32_t prmt0(uint32_t a, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(0u), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Per-lane constants of the scale/min decode for chunk c (sub-blocks 2c and
// 2c+1).  In the 12 packed bytes s[0..11] of the GGUF Q4_K layout, sub-block
// j < 4 has sc = s[j] & 63, m = s[j+4] & 63; j >= 4 has
// sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4.
// Both sub-blocks of a chunk read the byte pair at offset p = 2(c & 1) of
// s[0..3], s[4..7], s[8..11]; `sel` moves that pair into the two 16-bit
// halves of a word, and the masks keep the fields of the lane's case.
struct LaneDec {
  uint32_t sel, ma, mb, mc;
};
__device__ __forceinline__ LaneDec lane_dec(int c) {
  LaneDec L;
  L.sel = (c & 1) ? 0x4342u : 0x4140u;
  const bool hi = c >= 2;
  L.ma = hi ? 0u : 0x003F003Fu;
  L.mb = hi ? 0x000F000Fu : 0u;
  L.mc = hi ? 0x00300030u : 0u;
  return L;
}

// acc += s0*p0 + s1*p1 + t0*x0 + t1*x1 where s = d * (sc_lo, sc_hi/16) and
// t = dmin * (-m_lo, -m_hi) are exact fp16 x fp16 products in fp32.
__device__ __forceinline__ void scale_acc(float& acc, uint32_t dd, uint32_t sc2, uint32_t nm2, float p0, float p1,
                                          float x0, float x1) {
  asm("{\n .reg .b16 d0, d1, s0, s1, m0, m1;\n .reg .f32 a, b, e, f;\n"
      " mov.b32 {d0, d1}, %1;\n mov.b32 {s0, s1}, %2;\n mov.b32 {m0, m1}, %3;\n"
      " fma.rn.f32.f16 a, d0, s0, %8;\n fma.rn.f32.f16 b, d0, s1, %8;\n"
      " fma.rn.f32.f16 e, d1, m0, %8;\n fma.rn.f32.f16 f, d1, m1, %8;\n"
      " fma.rn.f32 %0, a, %4, %0;\n fma.rn.f32 %0, b, %5, %0;\n"
      " fma.rn.f32 %0, e, %6, %0;\n fma.rn.f32 %0, f, %7, %0;\n}"
      : "+f"(acc)
      : "r"(dd), "r"(sc2), "r"(nm2), "f"(p0), "f"(p1), "f"(x0), "f"(x1), "f"(0.f));
}

// acc += 2^-24 * (partial dot product of one lane's chunk (64 weights) of one
// block row); Xlo, Xhi are the chunk's two x sums times 2^-24.
__device__ __forceinline__ void chunk_dot(float& acc, const RowData& d, const uint4 (&xv)[8], float Xlo, float Xhi,
                                          const LaneDec& L) {
  const uint32_t qw[8] = {d.q0.x, d.q0.y, d.q0.z, d.q0.w, d.q1.x, d.q1.y, d.q1.z, d.q1.w};
  float alo0 = 0.f, alo1 = 0.f, ahi0 = 0.f, ahi1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = qw[i];
    const uint32_t w8 = w >> 8;
    const uint32_t l02 = w & 0x000F000Fu;   // q*2^-24   (bytes 0,2 low nibbles, fp16 subnormals)
    const uint32_t l13 = w8 & 0x000F000Fu;  // q*2^-24   (bytes 1,3 low)
    const uint32_t h02 = w & 0x00F000F0u;   // 16q*2^-24 (bytes 0,2 high)
    const uint32_t h13 = w8 & 0x00F000F0u;  // 16q*2^-24 (bytes 1,3 high)
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
  // Scales and mins of sub-blocks 2c (lo half) and 2c+1 (hi half), as fp16
  // 1024+v, then exact fp16 values: (sc_lo, sc_hi/16) and (-m_lo, -m_hi).
  const uint32_t py = prmt0(d.h.y, L.sel), pz = prmt0(d.h.z, L.sel), pw = prmt0(d.h.w, L.sel);
  uint32_t scw = lop3_and_or(py, L.ma, 0x64006400u);
  scw = lop3_and_or(pw, L.mb, scw);
  scw = lop3_and_or(py >> 2, L.mc, scw);
  uint32_t mw = lop3_and_or(pz, L.ma, 0x64006400u);
  mw = lop3_and_or(pw >> 4, L.mb, mw);
  mw = lop3_and_or(pz >> 2, L.mc, mw);
  const uint32_t sc2 = hfma2_bits(scw, 0x2C003C00u, 0xD400E400u);  // * (1, 1/16) + (-1024, -64)
  const uint32_t nm2 = hfma2_bits(mw, 0xBC00BC00u, 0x64006400u);   // * (-1, -1) + (1024, 1024)
  //   2^-24 sum_i w_i x_i = d*sc_lo * A_lo + d*sc_hi/16 * A_hi
  //                         - dmin*m_lo * X_lo - dmin*m_hi * X_hi      (A, X scaled by 2^-24)
  scale_acc(acc, d.h.x, sc2, nm2, alo0 + alo1, ahi0 + ahi1, Xlo, Xhi);
}

// Exact power-of-two scalings of the subnormal-code dot product.
constexpr float kTwoM24 = 5.9604644775390625e-8f;  // 2^-24
constexpr float kTwo24 = 16777216.0f;              // 2^24

}  // namespace
}  // namespace jllm

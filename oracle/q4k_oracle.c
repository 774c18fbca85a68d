/*
 * Q4_K oracle: a plain, slow, single-threaded CPU statement of what the
 * dequant-fused matmul computes.  TEST INFRASTRUCTURE ONLY: the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg use it; the GPU
 * library never links, calls or includes it, and it shares no source with the
 * CUDA path.
 *
 * What is defined where:
 *   - The operation Y[M,N] = X[M,K] * dequant(W)[N,K]^T, the op order
 *     d*sc*q - dmin*m and the per-element error bound
 *     |y - y_ref| <= 2e-3 * sum_k |x_k * w_nk| + 1e-5 specify this library's
 *     matmul.  It is the work of the "INT4 dequant-fused GEMV" (decode) and
 *     the "tensor-core MMQ Q4_K prefill" kernels that the genie-ai-runtime
 *     README lists under "At a glance" (Kernels bullet) and "Project layout"
 *     (src/kernels/).
 *   - The pages only say the runtime loads "GGUF only" models (README,
 *     "At a glance", Models bullet) and runs Qwen3-4B Q4_K_M.  The bit layout
 *     of a Q4_K super-block is NOT printed on the pages; it is the public GGUF
 *     Q4_K block format, restated below in our own words:
 *       bytes   0..1   d     (IEEE binary16, little endian)
 *       bytes   2..3   dmin  (IEEE binary16, little endian)
 *       bytes   4..15  s[0..11]: eight 6-bit scales sc_j and eight 6-bit mins m_j
 *                      j<4 : sc_j = s[j] & 63,            m_j = s[j+4] & 63
 *                      j>=4: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4
 *                            m_j  = (s[j+4] >> 4) | (s[j]   >> 6) << 4
 *       bytes  16..143 qs[0..127]: 4-bit codes.  For chunk c in 0..3 and
 *                      l in 0..31, weight 64c+l is the low nibble of
 *                      qs[32c+l] (sub-block 2c) and weight 64c+32+l is its
 *                      high nibble (sub-block 2c+1).
 *       value of weight i in sub-block j:  w = d*sc_j*q - dmin*m_j
 *
 * Precision.  Every quantity is formed in fp64.  For finite fp16 d and dmin,
 * d*sc*q and dmin*m are integers times 2^-24 below 2^26, so the fp64
 * difference is the exact real value.  The fp32 dequant is that exact value
 * rounded once to fp32 (round to nearest even), which is what an fp32
 * evaluation in the stated op order gives, since its three products are exact
 * in fp32.  The fp16 dequant is the fp32 value rounded to fp16 (nearest
 * even), by this file's own conversion routine.
 *
 * Pins (tests/test_oracle_pins.py): exhaustive fp16 decode against numpy,
 * fp32->fp16 rounding against numpy, single-bit probes of the 12 scale bytes
 * and of the 128 code bytes against hand-written tables from the format
 * definition, the closed-form blocks (all-zero codes give -dmin*m_j; q=15,
 * sc=63 gives 15*63*d - dmin*m), a quantise->dequantise round trip, brute
 * force dot products, identity/ones/linearity probes of the matmul.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (no FMA contraction, so every
 * fp64 operation rounds as written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 256          /* weights per super-block                 */
#define BLOCK_BYTES 144 /* bytes per super-block                   */

/* ---------------------------------------------------------------- fp16 --- */

/* IEEE binary16 bits -> double, exactly (every binary16 value is a double). */
double oq_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int f = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* fp32 -> IEEE binary16 bits, round to nearest, ties to even. */
uint16_t oq_float_to_half_rne(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ax = x & 0x7fffffffu;
  if (ax >= 0x7f800000u) { /* inf or nan */
    if (ax == 0x7f800000u) return sign | 0x7c00u;
    return sign | 0x7e00u | (uint16_t)((ax >> 13) & 0x3ffu);
  }
  if (ax >= 0x477ff000u) return sign | 0x7c00u; /* >= 65520 rounds to inf */
  uint32_t e = ax >> 23;
  uint32_t mant = ax & 0x7fffffu;
  if (e < 113) { /* below 2^-14: binary16 subnormal or zero */
    if (e == 0) return sign; /* fp32 zero/subnormal is far below 2^-25 */
    mant |= 0x800000u;
    uint32_t shift = 126 - e; /* value = mant * 2^(e-150); unit 2^-24 */
    if (shift > 24) return sign;
    uint32_t q = mant >> shift;
    uint32_t rem = mant & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return sign | (uint16_t)q;
  }
  uint32_t q = ((e - 112) << 10) | (mant >> 13);
  uint32_t rem = mant & 0x1fffu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
  return sign | (uint16_t)q;
}

/* ---------------------------------------------------------- Q4_K block --- */

/* The 6-bit scale sc_j and min m_j of sub-block j (format table above). */
void oq_scale_min(const uint8_t s[12], int j, int* sc, int* m) {
  if (j < 4) {
    *sc = s[j] & 63;
    *m = s[j + 4] & 63;
  } else {
    *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
    *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
}

/* Inverse of oq_scale_min: pack eight (sc_j, m_j) pairs, each 0..63. */
void oq_pack_scale_min(const int sc[8], const int m[8], uint8_t s[12]) {
  for (int j = 0; j < 4; j++) {
    s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
    s[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
    s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
  }
}

/* 4-bit code of weight i (0..255) of a block. */
static int code_of(const uint8_t* qs, int i) {
  int c = i / 64, r = i % 64;
  uint8_t byte = qs[32 * c + (r % 32)];
  return r < 32 ? (byte & 15) : (byte >> 4);
}

/* Decode one 144-byte block into its 256 exact values. */
void oq_decode_block(const uint8_t* blk, double out[QK]) {
  double d = oq_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
  double dmin = oq_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
  const uint8_t* s = blk + 4;
  const uint8_t* qs = blk + 16;
  for (int i = 0; i < QK; i++) {
    int j = i / 32, sc, m;
    oq_scale_min(s, j, &sc, &m);
    double q = (double)code_of(qs, i);
    out[i] = d * (double)sc * q - dmin * (double)m;
  }
}

/* Decode row n of W ([N][K/256] blocks) into K exact values. */
void oq_decode_row(const uint8_t* w, int64_t K, int64_t n, double* row) {
  int64_t nb = K / QK;
  for (int64_t b = 0; b < nb; b++)
    oq_decode_block(w + (n * nb + b) * BLOCK_BYTES, row + b * QK);
}

/* dequant(W) as [N,K] row-major; out_dtype 0 = fp32, 1 = fp16 bits. */
void oq_dequant(const uint8_t* w, int64_t N, int64_t K, int out_dtype, void* out) {
  double blk[QK];
  int64_t nb = K / QK;
  for (int64_t n = 0; n < N; n++) {
    for (int64_t b = 0; b < nb; b++) {
      oq_decode_block(w + (n * nb + b) * BLOCK_BYTES, blk);
      for (int i = 0; i < QK; i++) {
        int64_t idx = n * K + b * QK + i;
        float v32 = (float)blk[i]; /* one rounding of the exact value */
        if (out_dtype == 0)
          ((float*)out)[idx] = v32;
        else
          ((uint16_t*)out)[idx] = oq_float_to_half_rne(v32);
      }
    }
  }
}

/* -------------------------------------------------------------- matmul --- */

/* y[m,n] = sum_k x[m,k] * W[n,k] and s[m,n] = sum_k |x[m,k] * W[n,k]|, fp64,
 * k ascending, for every (m, n).  x is fp64 [M,K]. */
int oq_matmul(const uint8_t* w, const double* x, int64_t M, int64_t N, int64_t K,
              double* y, double* s) {
  double* row = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  if (!row) return -1;
  for (int64_t n = 0; n < N; n++) {
    oq_decode_row(w, K, n, row);
    for (int64_t m = 0; m < M; m++) {
      const double* xm = x + m * K;
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; k++) {
        double p = xm[k] * row[k];
        acc += p;
        mag += fabs(p);
      }
      y[m * N + n] = acc;
      if (s) s[m * N + n] = mag;
    }
  }
  free(row);
  return 0;
}

/* The same for a subset of output columns n = cols[c]; results are
 * [M][ncols] (column c of y holds output column cols[c]). */
int oq_matmul_cols(const uint8_t* w, const double* x, int64_t M, int64_t K,
                   const int64_t* cols, int64_t ncols, double* y, double* s) {
  double* row = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  if (!row) return -1;
  for (int64_t c = 0; c < ncols; c++) {
    oq_decode_row(w, K, cols[c], row);
    for (int64_t m = 0; m < M; m++) {
      const double* xm = x + m * K;
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; k++) {
        double p = xm[k] * row[k];
        acc += p;
        mag += fabs(p);
      }
      y[m * ncols + c] = acc;
      if (s) s[m * ncols + c] = mag;
    }
  }
  free(row);
  return 0;
}

/* --------------------------------------------------------------- SwiGLU --- */

/* h = silu(g) * u with silu(z) = z / (1 + e^-z), fp64. */
void oq_swiglu(const double* g, const double* u, int64_t n, double* h) {
  for (int64_t i = 0; i < n; i++) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* -------------------------------------------------------------- RMSNorm --- */

/* xn[m][k] = x[m][k] * gamma[k] / sqrt(mean_k x[m][k]^2 + eps) for each of the
 * M rows of K values, fp64, k ascending (the "RMSNorm" of the README's "fused
 * RMSNorm + RoPE + SwiGLU" kernel; the formula is the standard root-mean-square
 * layer norm, which the pages name but do not print). */
void oq_rmsnorm(const double* x, const double* gamma, int64_t M, int64_t K, double eps, double* xn) {
  for (int64_t m = 0; m < M; m++) {
    const double* xr = x + m * K;
    double ss = 0.0;
    for (int64_t k = 0; k < K; k++) ss += xr[k] * xr[k];
    const double r = 1.0 / sqrt(ss / (double)K + eps);
    for (int64_t k = 0; k < K; k++) xn[m * K + k] = xr[k] * r * gamma[k];
  }
}

/* ----------------------------------------------------------------- RoPE --- */

/* Rotary position embedding of n_heads head vectors of head_dim values each
 * (head_dim even, half = head_dim/2), at position pos, fp64: the "RoPE" of the
 * README's "fused RMSNorm + RoPE + SwiGLU" kernel.  The pages print neither
 * the pairing nor the frequencies; this is the form used by Qwen3 (the model
 * the pages run): value i of a head is paired with value i + half, the pair
 * is rotated by the angle pos * theta_i with theta_i = base^(-2i/head_dim):
 *   out[i]        = v[i] * cos(a) - v[i + half] * sin(a)
 *   out[i + half] = v[i + half] * cos(a) + v[i] * sin(a)
 * in_place allowed (out == v). */
void oq_rope(const double* v, int64_t n_heads, int64_t head_dim, int64_t pos, double base, double* out) {
  const int64_t half = head_dim / 2;
  for (int64_t h = 0; h < n_heads; h++) {
    const double* vh = v + h * head_dim;
    double* oh = out + h * head_dim;
    for (int64_t i = 0; i < half; i++) {
      const double theta = pow(base, -2.0 * (double)i / (double)head_dim);
      const double a = (double)pos * theta;
      const double c = cos(a), sn = sin(a);
      const double x0 = vh[i], x1 = vh[i + half];
      oh[i] = x0 * c - x1 * sn;
      oh[i + half] = x1 * c + x0 * sn;
    }
  }
}

/* ------------------------------------------------------- INT8 KV codec --- */

/* The "FP16 <-> INT8 KV convert" of the README (At a glance, KV cache bullet:
 * INT8 by default with "FP16-ULP-bounded drift"; Project layout, src/kernels/).
 * The pages give neither the scale granularity nor the rounding.  Reading:
 * one scale per vector of `dim` fp16 values (one head of one token), symmetric,
 * the scale a power of two s = 2^e stored as fp16:
 *   amax = max |v|;  e = the smallest integer with amax <= 127 * 2^e, clamped
 *   to [-24, 9] (e = -24 also for amax = 0);
 *   q = round-half-even(v / 2^e), clamped to [-127, 127];  decode v' = q * 2^e.
 * q * 2^e is exactly representable in fp16 for every such e and q, so decode is
 * exact and encode(decode(encode(v))) == encode(v): a second round trip does
 * not move any value (no drift at all, the strongest form of a drift bound).
 * The round trip moves each value by at most 2^e / 2 (2^e once the code
 * saturates, which only happens for amax above 127.5 * 2^9 = 65280). */
static int kv_exponent(double amax) {
  int e = -24;
  while (e < 9 && amax > 127.0 * ldexp(1.0, e)) e++;
  return e;
}

void oq_kv_encode(const uint16_t* v, int64_t n_vec, int64_t dim, int8_t* q, uint16_t* scale) {
  for (int64_t i = 0; i < n_vec; i++) {
    const uint16_t* vi = v + i * dim;
    double amax = 0.0;
    for (int64_t k = 0; k < dim; k++) {
      double a = fabs(oq_half_to_double(vi[k]));
      if (a > amax) amax = a;
    }
    const int e = kv_exponent(amax);
    const double s = ldexp(1.0, e);
    for (int64_t k = 0; k < dim; k++) {
      double t = oq_half_to_double(vi[k]) / s; /* exact: a power-of-two scaling */
      double r = nearbyint(t);                 /* round half to even (default mode) */
      if (r > 127.0) r = 127.0;
      if (r < -127.0) r = -127.0;
      q[i * dim + k] = (int8_t)r;
    }
    scale[i] = oq_float_to_half_rne((float)s); /* 2^e, exact in fp16 */
  }
}

void oq_kv_decode(const int8_t* q, const uint16_t* scale, int64_t n_vec, int64_t dim, uint16_t* out) {
  for (int64_t i = 0; i < n_vec; i++) {
    const double s = oq_half_to_double(scale[i]);
    for (int64_t k = 0; k < dim; k++) out[i * dim + k] = oq_float_to_half_rne((float)((double)q[i * dim + k] * s));
  }
}

/* ------------------------------------------------------------ quantiser --- */

/* Smallest binary16 value >= v (v >= 0, finite, below 65504), as bits. */
static uint16_t half_ceil(double v) {
  uint16_t h = oq_float_to_half_rne((float)v);
  while (oq_half_to_double(h) < v) h++; /* next binary16 up (v >= 0) */
  return h;
}

/* Quantise 256 values into one block, non-iteratively:
 *   per sub-block j: lo = min(0, min w), hi = max w, scale_j = (hi-lo)/15,
 *   off_j = -lo; d = smallest fp16 >= max scale_j / 63, dmin likewise for
 *   off_j; sc_j = ceil(scale_j / d), m_j = round(off_j / dmin) (both capped
 *   at 63); q = clamp(round((w + dmin*m_j) / (d*sc_j)), 0, 15).
 * Every decoded value lies within max(d*sc_j, dmin)/2 of its input. */
void oq_quantize_block(const double in[QK], uint8_t blk[BLOCK_BYTES]) {
  double scale[8], off[8], max_scale = 0.0, max_off = 0.0;
  for (int j = 0; j < 8; j++) {
    double lo = 0.0, hi = in[32 * j];
    for (int i = 0; i < 32; i++) {
      double v = in[32 * j + i];
      if (v < lo) lo = v;
      if (v > hi) hi = v;
    }
    if (hi < lo) hi = lo;
    scale[j] = (hi - lo) / 15.0;
    off[j] = -lo;
    if (scale[j] > max_scale) max_scale = scale[j];
    if (off[j] > max_off) max_off = off[j];
  }
  uint16_t dh = half_ceil(max_scale / 63.0), mh = half_ceil(max_off / 63.0);
  double d = oq_half_to_double(dh), dmin = oq_half_to_double(mh);
  int sc[8], m[8];
  for (int j = 0; j < 8; j++) {
    double a = d > 0.0 ? ceil(scale[j] / d) : 0.0;
    double b = dmin > 0.0 ? floor(off[j] / dmin + 0.5) : 0.0;
    sc[j] = a > 63.0 ? 63 : (int)a;
    m[j] = b > 63.0 ? 63 : (int)b;
  }
  memset(blk, 0, BLOCK_BYTES);
  blk[0] = (uint8_t)(dh & 255);
  blk[1] = (uint8_t)(dh >> 8);
  blk[2] = (uint8_t)(mh & 255);
  blk[3] = (uint8_t)(mh >> 8);
  oq_pack_scale_min(sc, m, blk + 4);
  uint8_t* qs = blk + 16;
  for (int i = 0; i < QK; i++) {
    int j = i / 32;
    double step = d * (double)sc[j];
    int q = 0;
    if (step > 0.0) {
      double t = floor((in[i] + dmin * (double)m[j]) / step + 0.5);
      q = t < 0.0 ? 0 : (t > 15.0 ? 15 : (int)t);
    }
    int c = i / 64, r = i % 64;
    if (r < 32)
      qs[32 * c + r] |= (uint8_t)q;
    else
      qs[32 * c + r - 32] |= (uint8_t)(q << 4);
  }
}

/* Quantise a [N,K] fp64 matrix block by block (oq_quantize_block). */
void oq_quantize(const double* w, int64_t N, int64_t K, uint8_t* out) {
  int64_t nb = K / QK;
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < nb; b++)
      oq_quantize_block(w + n * K + b * QK, out + (n * nb + b) * BLOCK_BYTES);
}

/* ------------------------------------------------ array forms (loops) --- */

void oq_half_to_double_n(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oq_half_to_double(h[i]);
}

void oq_float_to_half_rne_n(const float* f, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oq_float_to_half_rne(f[i]);
}

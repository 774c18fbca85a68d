"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a library routine, a
hand-written table of the GGUF Q4_K format, a closed form, an invariant or a
brute-force computation written independently here, chosen so that a plausible
slip in the oracle (a dropped term, a wrong sign, a swapped index or byte)
fails at least one of them.  CPU only.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _block(d_bits=0, dmin_bits=0, scales=None, qs=None):
    b = np.zeros(144, dtype=np.uint8)
    b[0], b[1] = d_bits & 255, d_bits >> 8
    b[2], b[3] = dmin_bits & 255, dmin_bits >> 8
    if scales is not None:
        b[4:16] = np.asarray(scales, dtype=np.uint8)
    if qs is not None:
        b[16:144] = np.asarray(qs, dtype=np.uint8)
    return b


def _h(v):
    """binary16 bits of a value exactly representable in fp16 (numpy)."""
    return int(np.array([v], dtype="<f2").view(np.uint16)[0])


# ------------------------------------------------------------------ fp16 ----

def test_half_decode_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.half_bits_to_double(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_float_to_half_rounding_against_numpy():
    rng = np.random.Generator(np.random.PCG64(7))
    parts = [
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(200000) * 1e-5).astype(np.float32),  # fp16 subnormal range
        (rng.standard_normal(50000) * 3e4).astype(np.float32),  # near overflow
        rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]
    # exact ties between neighbouring fp16 values (normal and subnormal)
    h = np.arange(0, 0x7bff, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    parts.append(((lo + hi) / 2).astype(np.float32))
    parts.append(np.array([65504.0, 65519.99, 65520.0, 1e9, np.inf, -np.inf, 0.0, -0.0,
                           2.0**-25, 2.0**-25 * 1.0000001, 3 * 2.0**-25, 2.0**-24], dtype=np.float32))
    f = np.concatenate(parts)
    f = f[~np.isnan(f)]
    got = oracle.float_to_half_bits(f)
    with np.errstate(over="ignore"):
        want = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


# ---------------------------------------------------------- block layout ----

def test_scale_bits_match_format_table():
    """Setting one of the 96 scale bits moves exactly the field the table names."""
    table = _read_table("q4k_scale_layout.txt")
    expect = {}
    for byte, blo, bhi, field, sub, shift in table:
        for b in range(int(blo), int(bhi) + 1):
            expect[(int(byte), b)] = (field, int(sub), 1 << (b - int(blo) + int(shift)))
    assert len(expect) == 96
    for (byte, bit), (field, sub, val) in expect.items():
        s = np.zeros(12, dtype=np.uint8)
        s[byte] = 1 << bit
        fields = {}
        for j in range(8):
            sc, m = oracle.scale_min(s, j)
            fields[("sc", j)] = sc
            fields[("m", j)] = m
        nonzero = {k: v for k, v in fields.items() if v}
        assert nonzero == {(field, sub): val}, (byte, bit, nonzero)


def test_scale_pack_inverts_unpack_exhaustively_per_slot():
    rng = np.random.Generator(np.random.PCG64(11))
    for j in range(8):
        for sc in range(64):
            for m in range(64):
                scs = rng.integers(0, 64, 8)
                ms = rng.integers(0, 64, 8)
                scs[j], ms[j] = sc, m
                s = oracle.pack_scale_min(scs, ms)
                for jj in range(8):
                    assert oracle.scale_min(s, jj) == (scs[jj], ms[jj])


def test_code_positions_match_format_table():
    """A single code of 1 (d=1, every sc=63, dmin=0) lights exactly the weight the table names."""
    table = _read_table("q4k_code_layout.txt")
    where = {}
    for first, last, nib, w0 in table:
        for t in range(int(last) - int(first) + 1):
            where[(int(first) + t, nib)] = int(w0) + t
    assert sorted(where.values()) == list(range(256))
    for (byte, nib), widx in where.items():
        qs = np.zeros(128, dtype=np.uint8)
        qs[byte] = 1 if nib == "low" else 16
        vals = oracle.decode_block(_block(_h(1.0), 0, [0xFF] * 12, qs))
        want = np.zeros(256)
        want[widx] = 63.0
        assert np.array_equal(vals, want), (byte, nib)


# ------------------------------------------------------------ closed forms ----

@pytest.mark.parametrize("d,dmin", [(1.0, 0.5), (2.0**-12, 2.0**-8), (0.0078125, 0.000244140625), (3.25, 0.0)])
def test_closed_form_all_fields_max(d, dmin):
    """All scale bits set gives sc_j = m_j = 63: q=15 -> 15*63*d - 63*dmin, q=0 -> -63*dmin."""
    hi = oracle.decode_block(_block(_h(d), _h(dmin), [0xFF] * 12, [0xFF] * 128))
    lo = oracle.decode_block(_block(_h(d), _h(dmin), [0xFF] * 12, [0x00] * 128))
    assert np.all(hi == 15 * 63 * d - 63 * dmin)
    assert np.all(lo == -63 * dmin)


def test_closed_form_zero_codes_give_minus_dmin_m():
    """sc_j = 0 and m_j = j+1 (bytes chosen by hand): every weight of sub-block j is -dmin*(j+1)."""
    scales = [0, 0, 0, 0, 1, 2, 3, 4, 0x50, 0x60, 0x70, 0x80]
    dmin = 0.0625
    for qs in ([0] * 128, list(range(128))):
        v = oracle.decode_block(_block(_h(0.5), _h(dmin), scales, qs))
        for j in range(8):
            assert np.all(v[32 * j:32 * j + 32] == -dmin * (j + 1))
    # codes zero and arbitrary scales: still -dmin*m_j
    scales2 = [0x3F, 0x15, 0x2A, 0x01, 1, 2, 3, 4, 0x5F, 0x6F, 0x7F, 0x8F]
    v = oracle.decode_block(_block(_h(0.5), _h(dmin), scales2, [0] * 128))
    for j in range(8):
        assert np.all(v[32 * j:32 * j + 32] == -dmin * (j + 1))


def test_closed_form_zero_d_dmin_gives_zero():
    rng = np.random.Generator(np.random.PCG64(3))
    blk = rng.integers(0, 256, 144, dtype=np.uint8)
    blk[0:4] = 0
    assert np.all(oracle.decode_block(blk) == 0.0)


def test_closed_form_mixed_scales_and_codes():
    """Hand-chosen fields: sc_j = 2j+1, m_j = 7-j; codes q = weight index % 16."""
    # bytes derived by hand from the bit table for sc = (1,3,5,7,9,11,13,15), m = (7..0)
    scales = [1, 3, 5, 7, 7, 6, 5, 4, 0x39, 0x2B, 0x1D, 0x0F]
    qs = np.zeros(128, dtype=np.uint8)
    for c in range(4):
        for l in range(32):
            lo_q = (64 * c + l) % 16
            hi_q = (64 * c + 32 + l) % 16
            qs[32 * c + l] = lo_q | (hi_q << 4)
    d, dmin = 0.25, 0.125
    v = oracle.decode_block(_block(_h(d), _h(dmin), scales, qs))
    for i in range(256):
        j = i // 32
        assert v[i] == d * (2 * j + 1) * (i % 16) - dmin * (7 - j)


def test_dequant_fp32_and_fp16_of_generated_weights():
    """fp32 output = exact value (exact in fp32 for d, dmin in [2^-12, 2^-8]); fp16 = numpy's rounding of it."""
    N, K = 16, 1024
    w = synthetic.q4k_weights(N, K, seed=5)
    exact = np.concatenate([oracle.decode_block(w[n, b * 144:(b + 1) * 144])
                            for n in range(N) for b in range(K // 256)]).reshape(N, K)
    f32 = oracle.dequant(w, N, K, "f32")
    assert np.array_equal(f32.astype(np.float64), exact)
    f16 = oracle.dequant(w, N, K, "f16")
    assert np.array_equal(f16.view(np.uint16), f32.astype(np.float16).view(np.uint16))


def test_dequant_fp32_rounds_once_for_wide_exponents():
    """d large, dmin tiny: the difference needs more than 24 bits and is rounded once to fp32."""
    blk = _block(_h(2048.0), _h(2.0**-24), [0xFF] * 12, [0x11] * 128)
    v = oracle.decode_block(blk)
    exact = 2048.0 * 63 * 1 - 2.0**-24 * 63
    assert np.all(v == exact)
    f32 = oracle.dequant(blk, 1, 256, "f32")
    assert np.all(f32 == np.float32(exact))
    assert float(np.float32(exact)) != exact


# ------------------------------------------------------------- round trip ----

def test_quantize_dequantize_round_trip_error():
    rng = np.random.Generator(np.random.PCG64(21))
    N, K = 8, 1024
    w = rng.standard_normal((N, K))
    q = oracle.quantize(w)
    back = _exact_w(q, N, K)
    err = back - w
    var_expect = []
    for n in range(N):
        for b in range(K // 256):
            blk = q[n, b * 144:(b + 1) * 144]
            d, dmin = oracle.half_bits_to_double(blk[0:4].copy().view("<u2"))
            for j in range(8):
                sc, _ = oracle.scale_min(blk[4:16], j)
                step = d * sc
                e = err[n, b * 256 + 32 * j: b * 256 + 32 * j + 32]
                assert np.all(np.abs(e) <= 0.5 * max(step, dmin) * (1 + 1e-9) + 1e-12)
                var_expect.append(step * step / 12.0)
    rms = math.sqrt(float(np.mean(err ** 2)))
    rms_expect = math.sqrt(float(np.mean(var_expect)))
    assert 0.75 * rms_expect <= rms <= 1.25 * rms_expect


def test_exact_codes_round_trip():
    """Blocks whose every sub-block uses q=0 and q=15, with max sc = max m = 63, come back exactly."""
    rng = np.random.Generator(np.random.PCG64(33))
    for trial in range(40):
        sc = rng.integers(1, 64, 8)
        m = rng.integers(0, 64, 8)
        sc[rng.integers(0, 8)] = 63
        m[rng.integers(0, 8)] = 63
        codes = rng.integers(0, 16, 256)
        for j in range(8):
            pos = rng.choice(32, 2, replace=False) + 32 * j
            codes[pos[0]], codes[pos[1]] = 0, 15
        qs = np.zeros(128, dtype=np.uint8)
        for i in range(256):
            c, r = divmod(i, 64)
            if r < 32:
                qs[32 * c + r] |= codes[i]
            else:
                qs[32 * c + r - 32] |= codes[i] << 4
        d = float(np.float16(rng.uniform(2**-12, 2**-8)))
        dmin = float(np.float16(rng.uniform(2**-12, 2**-8)))
        blk = _block(_h(d), _h(dmin), oracle.pack_scale_min(sc, m), qs)
        v = oracle.decode_block(blk)
        v2 = oracle.decode_block(oracle.quantize(v.reshape(1, 256)).reshape(144))
        assert np.array_equal(v, v2), trial


# ----------------------------------------------------------------- matmul ----

def _exact_w(w, N, K):
    return np.concatenate([oracle.decode_block(w[n, b * 144:(b + 1) * 144])
                           for n in range(N) for b in range(K // 256)]).reshape(N, K)


@pytest.mark.parametrize("M,N,K", [(1, 3, 256), (2, 5, 512), (5, 8, 256), (3, 1, 512)])
def test_matmul_brute_force_tiny(M, N, K):
    w = synthetic.q4k_weights(N, K, seed=100 + M * 10 + N)
    x = synthetic.activations(M, K, seed=200 + M)
    y, s = oracle.matmul(w, x, N, K)
    W = _exact_w(w, N, K)
    xd = x.astype(np.float64)
    for m in range(M):
        for n in range(N):
            terms = [float(xd[m, k]) * float(W[n, k]) for k in range(K)]
            ref = math.fsum(terms)
            mag = math.fsum(abs(t) for t in terms)
            assert abs(y[m, n] - ref) <= 1e-13 * mag + 1e-300
            assert abs(s[m, n] - mag) <= 1e-13 * mag


def test_matmul_unit_vectors_pick_columns():
    N, K = 6, 512
    w = synthetic.q4k_weights(N, K, seed=9)
    W = _exact_w(w, N, K)
    ks = [0, 1, 31, 32, 63, 64, 255, 256, 300, 511]
    x = np.zeros((len(ks), K))
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y, s = oracle.matmul(w, x, N, K)
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], W[:, k])
        assert np.array_equal(s[i], np.abs(W[:, k]))


def test_matmul_ones_gives_row_sums_and_linearity():
    N, K = 7, 768
    w = synthetic.q4k_weights(N, K, seed=10)
    W = _exact_w(w, N, K)
    y, _ = oracle.matmul(w, np.ones((1, K)), N, K)
    assert np.allclose(y[0], W.sum(axis=1), rtol=1e-14, atol=1e-14)
    x1 = synthetic.activations(2, K, seed=1).astype(np.float64)
    x2 = synthetic.activations(2, K, seed=2).astype(np.float64)
    a, b = 0.75, -2.5
    y1, s1 = oracle.matmul(w, x1, N, K)
    y2, s2 = oracle.matmul(w, x2, N, K)
    y3, _ = oracle.matmul(w, a * x1 + b * x2, N, K)
    assert np.all(np.abs(y3 - (a * y1 + b * y2)) <= 1e-13 * (abs(a) * s1 + abs(b) * s2))


def test_matmul_bound_and_cols_subset():
    N, K, M = 9, 512, 3
    w = synthetic.q4k_weights(N, K, seed=12)
    x = synthetic.activations(M, K, seed=13, per_token_scale=True)
    y, s = oracle.matmul(w, x, N, K)
    W = _exact_w(w, N, K)
    assert np.allclose(s, np.abs(x.astype(np.float64)) @ np.abs(W).T, rtol=1e-13)
    assert np.allclose(y, x.astype(np.float64) @ W.T, rtol=1e-12, atol=1e-12)
    cols = [8, 0, 4]
    yc, sc = oracle.matmul_cols(w, x, N, K, cols)
    assert np.array_equal(yc, y[:, cols])
    assert np.array_equal(sc, s[:, cols])


# ----------------------------------------------------------------- SwiGLU ----

def test_swiglu_against_closed_forms():
    scipy_special = pytest.importorskip("scipy.special")
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 800.0, -800.0, 2.5])
    u = np.array([3.0, 2.0, 2.0, 1.0, 1.0, 1.0, 1.0, -4.0])
    h = oracle.swiglu(g, u)
    assert h[0] == 0.0
    assert h[3] == pytest.approx(30.0, rel=1e-12)
    assert abs(h[4]) < 1e-11
    assert h[5] == 800.0 and h[6] == 0.0
    ref = g * scipy_special.expit(g) * u
    assert np.allclose(h, ref, rtol=1e-14, atol=1e-300)
    assert h[1] == pytest.approx(2.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


# ------------------------------------------------------- synthetic inputs ----

def test_swiglu_tolerance_covers_perturbed_inputs_and_is_not_loose():
    """swiglu_tolerance against what it claims to bound: h' = fp16(silu(g')*u') for every
    g', u' within the matmul bound of g, u (the four corners and random interior points of
    the box), computed in fp64 and rounded to fp16; and not loose where silu' >= 1/2 (the
    bound is within 3x of the largest deviation found there)."""
    rng = np.random.Generator(np.random.PCG64(3))
    n = 20000
    g = rng.normal(0.0, 4.0, n)
    u = rng.normal(0.0, 4.0, n)
    u[:200] *= 1e-3  # |u| far below its own bound: the perturbed product dominates
    sg = rng.uniform(0.0, 50.0, n)
    su = rng.uniform(0.0, 50.0, n)
    eg, eu = oracle.tolerance(sg), oracle.tolerance(su)
    h = oracle.swiglu(g, u)
    tol = oracle.swiglu_tolerance(g, u, sg, su)
    worst = np.zeros(n)
    deltas = [(a, b) for a in (-1.0, 1.0) for b in (-1.0, 1.0)]
    deltas += [tuple(rng.uniform(-1.0, 1.0, 2)) for _ in range(8)]
    for a, b in deltas:
        hp = oracle.swiglu(g + a * eg, u + b * eu).astype(np.float16).astype(np.float64)
        worst = np.maximum(worst, np.abs(hp - h))
    assert np.all(worst <= tol)
    sig = 1.0 / (1.0 + np.exp(-g))
    steep = sig * (1.0 + g * (1.0 - sig)) >= 0.5
    assert steep.sum() > 5000
    assert np.all(tol[steep] <= 3.0 * worst[steep])


def test_rmsnorm_against_closed_forms():
    # (3, 4): mean square 12.5, root 5/sqrt(2): outputs 3*sqrt(2)/5 and 4*sqrt(2)/5
    xn = oracle.rmsnorm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    assert np.allclose(xn, [3 * math.sqrt(2) / 5, 4 * math.sqrt(2) / 5], rtol=1e-15, atol=0)
    # a constant row normalises to its sign, whatever the constant (exactly for powers of two)
    for c in (-0.25, 4096.0):
        assert np.array_equal(oracle.rmsnorm(np.full(256, c), np.ones(256), 0.0), np.full(256, math.copysign(1.0, c)))
    for c in (-7.5, 0.001, 3e4):
        xn = oracle.rmsnorm(np.full(256, c), np.ones(256), 0.0)
        assert np.allclose(xn, math.copysign(1.0, c), rtol=1e-14, atol=0)
    # eps sits under the root: 1 / sqrt(1 + 3) = 0.5
    assert oracle.rmsnorm(np.array([1.0]), np.ones(1), 3.0)[0] == 0.5
    # an all-zero row stays zero (no 0/0) when eps > 0
    assert np.array_equal(oracle.rmsnorm(np.zeros(64), np.ones(64), 1e-6), np.zeros(64))


def test_rmsnorm_invariants():
    rng = np.random.Generator(np.random.PCG64(77))
    x = rng.standard_normal((5, 512)) * rng.uniform(0.1, 10.0, size=(5, 1))
    g = rng.uniform(-2.0, 2.0, size=512)
    one = oracle.rmsnorm(x, np.ones(512), 0.0)
    # unit root-mean-square per row with gamma = 1 and eps = 0
    assert np.allclose(np.mean(one**2, axis=1), 1.0, rtol=1e-13)
    # invariant to a positive scale of the row
    assert np.allclose(oracle.rmsnorm(x * 37.0, np.ones(512), 0.0), one, rtol=1e-13, atol=1e-15)
    # gamma scales each column
    assert np.allclose(oracle.rmsnorm(x, g, 0.0), one * g, rtol=1e-13, atol=1e-15)
    # rows are independent: the batch equals the row-by-row results
    for m in range(5):
        assert np.array_equal(oracle.rmsnorm(x[m:m + 1], g, 1e-6)[0], oracle.rmsnorm(x[m], g, 1e-6))


# ------------------------------------------------------------------- RoPE ----

QWEN3_ROPE_BASE = 1.0e6


def test_rope_identity_at_position_zero():
    rng = np.random.Generator(np.random.PCG64(80))
    v = rng.standard_normal((3, 128))
    assert np.array_equal(oracle.rope(v, 0, QWEN3_ROPE_BASE), v)  # cos 0 = 1, sin 0 = 0 exactly


def test_rope_unit_vectors_pin_pairing_sign_and_frequencies():
    # Pair i rotates (e_i, e_{i+64}) counter-clockwise by pos * base^(-i/64): e_i goes to
    # cos a * e_i + sin a * e_{i+64}, e_{i+64} to -sin a * e_i + cos a * e_{i+64}.
    # Frequency 0 is exactly 1 rad per position: cos 1 = 0.5403023058681398, sin 1 = 0.8414709848078965.
    e0 = np.zeros(128)
    e0[0] = 1.0
    r = oracle.rope(e0, 1, QWEN3_ROPE_BASE)
    assert r[0] == pytest.approx(0.5403023058681398, abs=1e-16)
    assert r[64] == pytest.approx(0.8414709848078965, abs=1e-16)
    assert np.count_nonzero(r) == 2
    for i, pos in ((1, 7), (32, 1000), (63, 32767)):
        a = pos * QWEN3_ROPE_BASE ** (-i / 64.0)
        for src, want in ((i, {i: math.cos(a), i + 64: math.sin(a)}), (i + 64, {i: -math.sin(a), i + 64: math.cos(a)})):
            v = np.zeros(128)
            v[src] = 1.0
            r = oracle.rope(v, pos, QWEN3_ROPE_BASE)
            for k, val in want.items():
                assert r[k] == pytest.approx(val, abs=1e-12), (i, pos, src, k)
            assert np.count_nonzero(r) <= 2
    # the lowest frequency with base 10^6 and head size 128: 10^(-6*63/64) rad per position
    v = np.zeros(128)
    v[63] = 1.0
    a = 1e5 * 10.0 ** (-6.0 * 63.0 / 64.0)
    assert oracle.rope(v, 100000, QWEN3_ROPE_BASE)[127] == pytest.approx(math.sin(a), abs=1e-12)


def test_rope_preserves_pair_norms_and_composes():
    rng = np.random.Generator(np.random.PCG64(81))
    v = rng.standard_normal((4, 128)) * 3.0
    r = oracle.rope(v, 12345, QWEN3_ROPE_BASE)
    n0 = v[:, :64] ** 2 + v[:, 64:] ** 2
    n1 = r[:, :64] ** 2 + r[:, 64:] ** 2
    assert np.allclose(n1, n0, rtol=1e-13, atol=1e-13)
    # rotation by p1 then p2 equals rotation by p1 + p2; by p then -p is the identity
    for p1, p2 in ((3, 5), (1000, 24), (20000, 12767)):
        a = oracle.rope(oracle.rope(v, p1, QWEN3_ROPE_BASE), p2, QWEN3_ROPE_BASE)
        b = oracle.rope(v, p1 + p2, QWEN3_ROPE_BASE)
        assert np.allclose(a, b, rtol=0, atol=1e-9)
    back = oracle.rope(oracle.rope(v, 777, QWEN3_ROPE_BASE), -777, QWEN3_ROPE_BASE)
    assert np.allclose(back, v, rtol=0, atol=1e-12)
    # heads are independent and linear: the rotation of a sum is the sum of rotations
    w = rng.standard_normal((4, 128))
    lhs = oracle.rope(v + 2.0 * w, 99, QWEN3_ROPE_BASE)
    rhs = oracle.rope(v, 99, QWEN3_ROPE_BASE) + 2.0 * oracle.rope(w, 99, QWEN3_ROPE_BASE)
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)


def test_head_rmsnorm_is_rmsnorm_per_head():
    rng = np.random.Generator(np.random.PCG64(82))
    v = rng.standard_normal(8 * 128) * np.repeat(rng.uniform(0.1, 10.0, size=8), 128)
    g = rng.uniform(0.5, 1.5, size=128)
    hn = oracle.head_rmsnorm(v, g, 1e-6).reshape(8, 128)
    for h in range(8):
        seg = v[h * 128:(h + 1) * 128]
        assert np.array_equal(hn[h], oracle.rmsnorm(seg, g, 1e-6))
        # unit root-mean-square per head before gamma (eps negligible here)
        assert np.mean((hn[h] / g) ** 2) == pytest.approx(1.0, rel=1e-5)


# ---------------------------------------------------------- INT8 KV codec ----

def _kv_vectors(rng, n, dim=128):
    """fp16 vectors over many magnitudes, with some subnormal-only and some near the top of fp16."""
    mag = 10.0 ** rng.uniform(-9, 4.5, size=(n, 1))
    v = np.clip(rng.standard_normal((n, dim)) * mag, -65504, 65504)
    return v.astype(np.float16)


def test_kv_scale_is_the_smallest_power_of_two_covering_the_vector():
    rng = np.random.Generator(np.random.PCG64(90))
    v = _kv_vectors(rng, 3000)
    q, s = oracle.kv_encode(v)
    amax = np.max(np.abs(v.astype(np.float64)), axis=1)
    for i in range(v.shape[0]):
        # brute force over every allowed exponent
        cands = [e for e in range(-24, 10) if amax[i] <= 127.0 * 2.0**e]
        e = cands[0] if cands else 9
        assert float(s[i]) == 2.0**e, (i, amax[i], float(s[i]))
    # unclamped vectors use codes up to 127 and at least 64 in magnitude
    inner = (amax > 127.0 * 2.0**-24) & (amax <= 127.0 * 2.0**9)
    qmax = np.max(np.abs(q.astype(np.int64)), axis=1)
    assert np.all((qmax[inner] >= 64) & (qmax[inner] <= 127))


def test_kv_closed_forms():
    # exact multiples of the scale come back exactly, codes = the multiples
    k = np.arange(-127, 129, dtype=np.int64)[:128]
    for e in (-24, -20, -3, 0, 5, 9):
        v = (k * 2.0**e).astype(np.float16)
        q, s = oracle.kv_encode(v[None, :])
        assert float(s[0]) == 2.0**e and np.array_equal(q[0].astype(np.int64), k)
        assert np.array_equal(oracle.kv_decode(q, s), v[None, :])
    # round half to even: 2.5 -> 2, 3.5 -> 4, -0.5 -> -0, with the scale pinned to 1 by 127
    v = np.zeros(128, dtype=np.float16)
    v[:4] = [127.0, 2.5, 3.5, -0.5]
    q, s = oracle.kv_encode(v[None, :])
    assert float(s[0]) == 1.0 and list(q[0, :4]) == [127, 2, 4, 0]
    # a zero vector stays zero; sign symmetry
    q0, s0 = oracle.kv_encode(np.zeros((1, 128), np.float16))
    assert not q0.any() and np.all(oracle.kv_decode(q0, s0) == 0)
    rng = np.random.Generator(np.random.PCG64(91))
    v = _kv_vectors(rng, 200)
    qa, sa = oracle.kv_encode(v)
    qb, sb = oracle.kv_encode(-v)
    assert np.array_equal(qb, -qa) and np.array_equal(sb, sa)
    # the top of the fp16 range saturates: 65504 / 512 = 127.94 -> 127, decoded 65024
    v = np.zeros((1, 128), np.float16)
    v[0, 0] = 65504.0
    q, s = oracle.kv_encode(v)
    assert float(s[0]) == 512.0 and q[0, 0] == 127 and float(oracle.kv_decode(q, s)[0, 0]) == 65024.0


def test_kv_round_trip_error_and_no_drift():
    rng = np.random.Generator(np.random.PCG64(92))
    v = _kv_vectors(rng, 4000)
    q, s = oracle.kv_encode(v)
    d = oracle.kv_decode(q, s)
    err = np.abs(d.astype(np.float64) - v.astype(np.float64))
    sf = s.astype(np.float64)[:, None]
    amax = np.max(np.abs(v.astype(np.float64)), axis=1)
    sat = (amax > 127.5 * 2.0**9)[:, None]
    assert np.all(err <= np.where(sat, sf, sf / 2))
    # decode is exact (q * 2^e in fp16) and a second round trip changes nothing
    assert np.array_equal(d.astype(np.float64), q.astype(np.float64) * sf)
    q2, s2 = oracle.kv_encode(d)
    assert np.array_equal(q2, q) and np.array_equal(s2, s)
    assert np.array_equal(oracle.kv_decode(q2, s2), d)
    # vectors whose values are all below 127 * 2^-24 (fp16 subnormal range) round-trip exactly
    tiny = (rng.integers(-127, 128, size=(50, 128)) * 2.0**-24).astype(np.float16)
    qt, st = oracle.kv_encode(tiny)
    assert np.all(st.astype(np.float64) == 2.0**-24) and np.array_equal(oracle.kv_decode(qt, st), tiny)


def test_synthetic_weights_distribution():
    w = synthetic.q4k_weights(64, 2560, seed=1)
    assert w.shape == (64, 10 * 144)
    blk = w.reshape(-1, 144)
    d = blk[:, 0:2].copy().view("<f2").astype(np.float64).ravel()
    dmin = blk[:, 2:4].copy().view("<f2").astype(np.float64).ravel()
    for v in (d, dmin):
        assert v.min() >= 2.0**-12 and v.max() <= 2.0**-8
        assert v.max() > 0.9 * 2.0**-8 and v.min() < 1.1 * 2.0**-12
    seen_sc, seen_m = set(), set()
    for b in blk[:200]:
        for j in range(8):
            sc, m = oracle.scale_min(b[4:16], j)
            seen_sc.add(sc)
            seen_m.add(m)
    assert seen_sc == set(range(64)) and seen_m == set(range(64))
    assert np.array_equal(w, synthetic.q4k_weights(64, 2560, seed=1))
    assert not np.array_equal(w, synthetic.q4k_weights(64, 2560, seed=2))


def test_synthetic_activations():
    x = synthetic.activations(4, 4096, seed=3)
    assert x.dtype == np.float16 and x.shape == (4, 4096)
    assert abs(float(x.astype(np.float64).mean())) < 0.05
    assert abs(float(x.astype(np.float64).std()) - 1.0) < 0.05
    xs = synthetic.activations(64, 1024, seed=4, per_token_scale=True).astype(np.float64)
    sd = xs.std(axis=1)
    assert sd.min() > 0.4 and sd.max() < 2.3

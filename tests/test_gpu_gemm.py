"""GPU GEMM (tcgen05 path for M above the GEMV threshold) vs the oracle."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import LAYER_SHAPES, assert_within, dev, sample_cols, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def _gemm(q, w_np, x_np, N, K, f16):
    import torch

    out = q.jllm_q4k_gemm(dev(w_np), dev(x_np), N, K, out_dtype=torch.float16 if f16 else torch.float32)
    return out.float().cpu().numpy()


# 129..256 with few weight-row tiles also covers the split into two token tiles;
# above 256 the wide tiles: one of 320 / 384 / 512 tokens (halves of 160..256,
# the second half cut short at 449 and 511), then two, three token tiles
@pytest.mark.parametrize("M", [2, 5, 16, 17, 33, 64, 100, 128, 129, 130, 200, 255, 256, 257, 300,
                               384, 449, 511, 512, 513, 700, 1025])
def test_gemm_small_full(q, M):
    N, K = 200, 768
    w = synthetic.q4k_weights(N, K, 900 + M)
    x = synthetic.activations(M, K, 950 + M, per_token_scale=True)
    ref, s = oracle.matmul(w, x, N, K)
    assert_within(_gemm(q, w, x, N, K, False), ref, s, f"M={M} f32")


@pytest.mark.parametrize("N,K,M", [(1, 256, 40), (129, 256, 3), (300, 1280, 70), (64, 9728, 20), (1000, 2560, 520)])
def test_gemm_ragged_full(q, N, K, M):
    w = synthetic.q4k_weights(N, K, 1100 + N)
    x = synthetic.activations(M, K, 1200 + M)
    ref, s = oracle.matmul(w, x, N, K)
    assert_within(_gemm(q, w, x, N, K, False), ref, s, f"N={N} K={K} M={M}")


def test_gemm_fp16_output(q):
    """fp16 output adds one rounding: bound 2e-3*S + 2^-11*|ref| + 1e-5 (+ subnormal step)."""
    N, K, M = 256, 2560, 64
    w = synthetic.q4k_weights(N, K, 1300)
    x = synthetic.activations(M, K, 1301)
    ref, s = oracle.matmul(w, x, N, K)
    y = _gemm(q, w, x, N, K, True).astype(np.float64)
    tol = oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24
    assert np.all(np.abs(y - ref) <= tol)


def test_gemm_unit_vectors_give_fp16_dequant(q):
    """x rows = unit vectors: y = fp16(w) exactly (fp16 W tile, one product, fp32 accumulation).
    80 tokens: the tcgen05 path (fewer tokens take the factored form of the few-token GEMM)."""
    N, K = 130, 512
    w = synthetic.q4k_weights(N, K, 1400)
    ks = np.array([0, 1, 2, 31, 32, 33, 63, 64, 100, 127, 128, 200, 255, 256, 300, 511] * 5)
    x = np.zeros((len(ks), K), dtype=np.float16)
    x[np.arange(len(ks)), ks] = 1.0
    W16 = oracle.dequant(w, N, K, "f16").astype(np.float32)
    y = _gemm(q, w, x, N, K, False)
    assert np.array_equal(y, W16[:, ks].T)


def test_gemm_rows_match_gemv(q):
    N, K, M = 512, 2560, 40
    w = synthetic.q4k_weights(N, K, 1500)
    x = synthetic.activations(M, K, 1501)
    ref, s = oracle.matmul(w, x, N, K)
    y = _gemm(q, w, x, N, K, False)
    wd = dev(w)
    for m in (0, 17, 39):
        g = q.jllm_q4k_gemv(wd, dev(x[m]), N, K).cpu().numpy()
        assert np.all(np.abs(g - y[m]) <= 2 * oracle.tolerance(s[m]))


def test_gemm_linearity(q):
    N, K, M = 256, 1024, 48
    w = synthetic.q4k_weights(N, K, 1600)
    x1 = synthetic.activations(M, K, 1601)
    x2 = synthetic.activations(M, K, 1602)
    a, b = 0.5, -0.25
    x3 = (a * x1.astype(np.float64) + b * x2.astype(np.float64)).astype(np.float16)
    y1, y2, y3 = (_gemm(q, w, xx, N, K, False).astype(np.float64) for xx in (x1, x2, x3))
    r1, s1 = oracle.matmul(w, x1, N, K)
    r2, s2 = oracle.matmul(w, x2, N, K)
    r3, s3 = oracle.matmul(w, x3, N, K)
    # y3 - (a*y1 + b*y2) differs from r3 - (a*r1 + b*r2) (the fp16 rounding of x3) by at most the three bounds
    bound = oracle.tolerance(s3) + abs(a) * oracle.tolerance(s1) + abs(b) * oracle.tolerance(s2)
    assert np.all(np.abs((y3 - (a * y1 + b * y2)) - (r3 - (a * r1 + b * r2))) <= bound)


@pytest.mark.parametrize("M", [33, 235])
@pytest.mark.parametrize("name,K,N", LAYER_SHAPES)
def test_gemm_short_prefill_shapes(q, name, K, N, M):
    idx = [s[0] for s in LAYER_SHAPES].index(name)
    w = synthetic.q4k_weights(N, K, synthetic.weight_seed(2, 0, idx))
    x = synthetic.activations(M, K, synthetic.activation_seed(2, M, idx), per_token_scale=True)
    y = _gemm(q, w, x, N, K, True)
    rng = np.random.Generator(np.random.PCG64(M * 100 + idx))
    cols = sample_cols(N, rng)
    ref, s = oracle.matmul_cols(w, x, N, K, cols)
    tol_extra = 2.0**-11 * np.abs(ref) + 2.0**-24
    err = np.abs(y[:, cols] - ref)
    assert np.all(err <= oracle.tolerance(s) + tol_extra), f"{name} M={M}"


@pytest.mark.parametrize("M", [1024, 2048, 3072])
@pytest.mark.parametrize("name,K,N", LAYER_SHAPES)
def test_gemm_long_prefill_shapes(q, name, K, N, M):
    idx = [s[0] for s in LAYER_SHAPES].index(name)
    w = synthetic.q4k_weights(N, K, synthetic.weight_seed(3, 0, idx))
    x = synthetic.activations(M, K, synthetic.activation_seed(3, M, idx))
    y = _gemm(q, w, x, N, K, True)
    rng = np.random.Generator(np.random.PCG64(M * 10 + idx))
    cols = sample_cols(N, rng, n_random=48, edge=16)
    rows = sample_rows(M, rng)
    ref, s = oracle.matmul_cols(w, x[rows], N, K, cols)
    got = y[np.ix_(rows, cols)]
    tol = oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24
    assert np.all(np.abs(got - ref) <= tol), f"{name} M={M}"
    assert np.all(np.isfinite(y))


def test_no_device_error_after_gemms(q):
    assert q.jllm_get_device_error() == q.JLLM_OK


def test_tensor_map_cache_keys_on_address_and_shape(q):
    """The GEMM reuses encoded tensor maps per (device, address, extents, box): the same buffer
    reused for new contents, a new buffer at a recycled address, and the same address seen with
    other extents must all compute the right product."""
    import torch

    K, M = 2560, 64
    x1 = synthetic.activations(M, K, 1500)
    big = synthetic.q4k_weights(384, K, 1501)
    wd = dev(big)
    for N in (384, 256, 130):  # one address, three row counts
        ref, s = oracle.matmul(big[:N], x1, N, K)
        y = q.jllm_q4k_gemm(wd[:N], dev(x1), N, K, out_dtype=torch.float32).cpu().numpy()
        assert_within(y, ref, s, f"N={N}")
    for seed in (1502, 1503):  # new contents in a buffer at (very likely) a recycled address
        del wd
        w = synthetic.q4k_weights(384, K, seed)
        wd = dev(w)
        xd = dev(synthetic.activations(M, K, seed + 10))
        ref, s = oracle.matmul(w, xd.cpu().numpy(), 384, K)
        y = q.jllm_q4k_gemm(wd, xd, 384, K, out_dtype=torch.float32).cpu().numpy()
        assert_within(y, ref, s, f"seed={seed}")

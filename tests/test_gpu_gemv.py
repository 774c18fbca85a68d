"""GPU GEMV (M = 1) vs the oracle: the matmul bound on every element, the
decode-sweep shapes in full, identity probes bit-exact, ragged shapes."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import LAYER_SHAPES, assert_within, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def _run(q, w_np, x_np, N, K):
    return q.jllm_q4k_gemv(dev(w_np), dev(x_np.reshape(K)), N, K).cpu().numpy().reshape(1, N)


def test_gemv_tiny_config(q):
    N, K = 256, 512
    w = synthetic.q4k_weights(N, K, synthetic.weight_seed(0, 0, 0))
    x = synthetic.activations(1, K, synthetic.activation_seed(0, 1))
    ref, s = oracle.matmul(w, x, N, K)
    assert_within(_run(q, w, x, N, K), ref, s, "tiny")


@pytest.mark.parametrize("layer", [0, 35])
@pytest.mark.parametrize("name,K,N", LAYER_SHAPES)
def test_gemv_decode_shapes(q, name, K, N, layer):
    idx = [s[0] for s in LAYER_SHAPES].index(name)
    w = synthetic.q4k_weights(N, K, synthetic.weight_seed(1, layer, idx))
    x = synthetic.activations(1, K, synthetic.activation_seed(1, 1, idx))
    ref, s = oracle.matmul(w, x, N, K)
    assert_within(_run(q, w, x, N, K), ref, s, f"{name} layer {layer}")


@pytest.mark.parametrize("N,K", [(1, 256), (3, 768), (5, 256), (129, 1280), (1000, 2560), (17, 9728), (64, 65536)])
def test_gemv_ragged(q, N, K):
    w = synthetic.q4k_weights(N, K, 500 + N)
    x = synthetic.activations(1, K, 600 + N)
    ref, s = oracle.matmul(w, x, N, K)
    assert_within(_run(q, w, x, N, K), ref, s, f"N={N} K={K}")


def test_gemv_unit_vectors_give_fp32_dequant_exactly(q):
    N, K = 96, 768
    w = synthetic.q4k_weights(N, K, 42)
    W32 = oracle.dequant(w, N, K, "f32")
    wd = dev(w)
    for k in (0, 1, 31, 32, 63, 64, 255, 256, 511, 767):
        x = np.zeros(K, dtype=np.float16)
        x[k] = 1.0
        y = q.jllm_q4k_gemv(wd, dev(x), N, K).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), W32[:, k].view(np.uint32)), k


def test_gemv_ones_and_zero(q):
    N, K = 200, 2560
    w = synthetic.q4k_weights(N, K, 43)
    ones = np.ones((1, K), dtype=np.float16)
    ref, s = oracle.matmul(w, ones, N, K)
    assert_within(_run(q, w, ones, N, K), ref, s, "ones")
    zero = np.zeros((1, K), dtype=np.float16)
    assert np.all(_run(q, w, zero, N, K) == 0.0)


def test_gemm_m1_is_gemv(q):
    import torch

    N, K = 1024, 2560
    w = dev(synthetic.q4k_weights(N, K, 44))
    x = dev(synthetic.activations(1, K, 45))
    a = q.jllm_q4k_gemv(w, x.view(K), N, K)
    b = q.jllm_q4k_gemm(w, x, N, K, out_dtype=torch.float32)
    assert q.jllm_q4k_gemv_max_m() >= 1
    assert torch.equal(a, b.view(N))


def test_gemv_repeatable(q):
    N, K = 4096, 2560
    w = dev(synthetic.q4k_weights(N, K, 46))
    x = dev(synthetic.activations(1, K, 47).reshape(K))
    a = q.jllm_q4k_gemv(w, x, N, K)
    b = q.jllm_q4k_gemv(w, x, N, K)
    assert np.array_equal(a.cpu().numpy(), b.cpu().numpy())

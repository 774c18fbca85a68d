"""Decode GEMV with the RMSNorm prologue (jllm_q4k_gemv_rmsnorm_batch): every output
within the matmul bound of the fp64 oracle applied to the fp64 RMS-normalised x."""
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


def _gamma(K, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.uniform(0.25, 2.0, size=K).astype(np.float32)


def _check(q, ws_np, Ns, K, x, gamma, eps, label):
    import torch

    ys = q.jllm_q4k_gemv_rmsnorm_batch([dev(w) for w in ws_np], dev(x), torch.from_numpy(gamma).cuda(), eps, Ns, K)
    xn = oracle.rmsnorm(x.astype(np.float64), gamma.astype(np.float64), eps)
    for i, (w, n) in enumerate(zip(ws_np, Ns)):
        ref, s = oracle.matmul(w, xn, n, K)
        assert_within(ys[i].cpu().numpy()[None, :], ref, s, f"{label}[{i}]")
    return ys


@pytest.mark.parametrize("group", [("q", "k", "v"), ("gate", "up")])
def test_norm_gemv_layer_groups(q, group):
    shapes = {name: (K, N, idx) for idx, (name, K, N) in enumerate(LAYER_SHAPES)}
    K = shapes[group[0]][0]
    Ns = [shapes[g][1] for g in group]
    ws_np = [synthetic.q4k_weights(shapes[g][1], K, synthetic.weight_seed(1, 0, shapes[g][2])) for g in group]
    x = synthetic.activations(1, K, 6100 + len(group))[0]
    _check(q, ws_np, Ns, K, x, _gamma(K, 6200), 1e-6, "+".join(group))
    assert q.jllm_get_device_error() == 0


@pytest.mark.parametrize("N,K", [(37, 512), (300, 9728), (129, 4096), (2560, 256)])
def test_norm_gemv_ragged_and_long_k(q, N, K):
    w = synthetic.q4k_weights(N, K, 6300 + N)
    x = synthetic.activations(1, K, 6400 + K)[0]
    _check(q, [w], [N], K, x, _gamma(K, 6500 + K), 1e-5, f"N={N} K={K}")


@pytest.mark.parametrize("scale", [1e-3, 1.0, 100.0])
def test_norm_gemv_scale_of_x(q, scale):
    """The norm removes the scale of x: outputs for c*x match the oracle (and each other)."""
    N, K = 512, 2560
    w = synthetic.q4k_weights(N, K, 6600)
    x = (synthetic.activations(1, K, 6601)[0].astype(np.float64) * scale).astype(np.float16)
    _check(q, [w], [N], K, x, _gamma(K, 6602), 1e-6, f"scale={scale}")


def test_norm_gemv_zero_x_and_determinism(q):
    import torch

    N, K = 256, 2560
    w = synthetic.q4k_weights(N, K, 6700)
    g = torch.from_numpy(_gamma(K, 6701)).cuda()
    y0 = q.jllm_q4k_gemv_rmsnorm_batch([dev(w)], torch.zeros(K, dtype=torch.float16, device="cuda"), g, 1e-6, [N], K)
    assert torch.count_nonzero(y0[0]) == 0
    x = dev(synthetic.activations(1, K, 6702)[0])
    a = q.jllm_q4k_gemv_rmsnorm_batch([dev(w)], x, g, 1e-6, [N], K)[0]
    b = q.jllm_q4k_gemv_rmsnorm_batch([dev(w)], x, g, 1e-6, [N], K)[0]
    assert torch.equal(a, b)
    assert q.jllm_get_device_error() == 0

"""GPU dequant vs the oracle: bit-exact in fp32 and fp16."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import LAYER_SHAPES, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def _check(q, w_np, N, K):
    import torch

    w = dev(w_np)
    for dt, name in ((torch.float32, "f32"), (torch.float16, "f16")):
        got = q.jllm_q4k_dequant(w, N, K, out_dtype=dt).cpu().numpy()
        want = oracle.dequant(w_np, N, K, name)
        view = np.uint32 if name == "f32" else np.uint16
        if not np.array_equal(got.view(view), want.view(view)):
            bad = np.argwhere(got.view(view) != want.view(view))
            raise AssertionError(f"{name} N={N} K={K}: {len(bad)} mismatches, first at {bad[0]}")


def test_dequant_tiny_config(q):
    N, K = 256, 512
    _check(q, synthetic.q4k_weights(N, K, synthetic.weight_seed(0, 0, 0)), N, K)


@pytest.mark.parametrize("name,K,N", LAYER_SHAPES)
def test_dequant_layer_shapes(q, name, K, N):
    idx = [s[0] for s in LAYER_SHAPES].index(name)
    _check(q, synthetic.q4k_weights(N, K, synthetic.weight_seed(1, 0, idx)), N, K)


@pytest.mark.parametrize("N,K", [(1, 256), (3, 768), (129, 256), (7, 4096)])
def test_dequant_ragged(q, N, K):
    _check(q, synthetic.q4k_weights(N, K, 1000 + N), N, K)


def test_dequant_arbitrary_finite_headers(q):
    """Any finite fp16 d/dmin (subnormal, negative, large): fp32 rounds once, fp16 from fp32."""
    rng = np.random.Generator(np.random.PCG64(77))
    N, K = 64, 1024
    w = rng.integers(0, 256, size=(N, K // 256, 144), dtype=np.uint8)
    bits = rng.integers(0, 0x7C00, size=(N, K // 256, 2), dtype=np.uint16)  # finite magnitudes
    bits |= (rng.integers(0, 2, size=bits.shape, dtype=np.uint16) << 15)  # random signs
    w[:, :, 0:4] = bits.astype("<u2").view(np.uint8).reshape(N, K // 256, 4)
    _check(q, w.reshape(N, -1), N, K)


def test_dequant_zero_and_extreme_blocks(q):
    N, K = 4, 256
    w = np.zeros((N, 144), dtype=np.uint8)
    w[1, 4:16] = 0xFF
    w[1, 16:] = 0xFF
    w[1, 0:4] = np.array([1.0, 0.5], dtype="<f2").view(np.uint8)
    w[2, 0:4] = np.array([65504.0, 2.0**-24], dtype="<f2").view(np.uint8)
    w[2, 4:] = 0xA5
    w[3, 0:4] = np.array([-3.0, -2.0**-14], dtype="<f2").view(np.uint8)
    w[3, 4:] = 0x5A
    _check(q, w, N, K)

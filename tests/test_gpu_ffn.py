"""Fused SwiGLU FFN block and LM head (gate/up 2560->9728 with silu(g)*u,
down 9728->2560, LM head 2560->151936) at M = 1 and M = 512, vs the oracle."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_within, dev, oracle_matmul_rows, sample_cols

pytestmark = pytest.mark.gpu

H, F, V = 2560, 9728, synthetic.LM_HEAD[2]


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


@pytest.fixture(scope="module")
def weights():
    return {
        "gate": synthetic.q4k_weights(F, H, synthetic.weight_seed(4, 0, 4)),
        "up": synthetic.q4k_weights(F, H, synthetic.weight_seed(4, 0, 5)),
        "down": synthetic.q4k_weights(H, F, synthetic.weight_seed(4, 0, 6)),
    }


def _check_h(h_gpu, wg, wu, x, N, K, cols=None):
    if cols is None:
        g, sg = oracle.matmul(wg, x, N, K)
        u, su = oracle.matmul(wu, x, N, K)
        h = h_gpu
    else:
        g, sg = oracle.matmul_cols(wg, x, N, K, cols)
        u, su = oracle.matmul_cols(wu, x, N, K, cols)
        h = h_gpu[:, cols]
    href = oracle.swiglu(g, u)
    tol = oracle.swiglu_tolerance(g, u, sg, su)
    err = np.abs(h.astype(np.float64) - href)
    assert np.all(err <= tol), f"max excess {(err - tol).max()}"
    return href


@pytest.mark.parametrize("M", [1, 2, 33])
def test_swiglu_small(q, M):
    N, K = 384, 1024
    wg = synthetic.q4k_weights(N, K, 2000)
    wu = synthetic.q4k_weights(N, K, 2001)
    x = synthetic.activations(M, K, 2002 + M)
    h = q.jllm_q4k_ffn_swiglu(dev(wg), dev(wu), dev(x), N, K).float().cpu().numpy()
    _check_h(h, wg, wu, x, N, K)


@pytest.mark.parametrize("M", [1, 512])
def test_ffn_block(q, weights, M):
    import torch

    x = synthetic.activations(M, H, synthetic.activation_seed(4, M))
    h = q.jllm_q4k_ffn_swiglu(dev(weights["gate"]), dev(weights["up"]), dev(x), F, H)
    hn = h.float().cpu().numpy()
    rng = np.random.Generator(np.random.PCG64(M))
    cols = None if M == 1 else sample_cols(F, rng)
    href = _check_h(hn, weights["gate"], weights["up"], x, F, H, cols)
    # down projection on the oracle's own fp16 h (computed from the oracle alone), every
    # token row; at M = 512 the oracle's h comes from row chunks on several host threads
    # and the down output is checked on sampled columns including the tail.
    if cols is None:
        h16 = href.astype(np.float16)
    else:
        g, _ = oracle_matmul_rows(weights["gate"], x, F, H)
        u, _ = oracle_matmul_rows(weights["up"], x, F, H)
        h16 = oracle.swiglu(g, u).astype(np.float16)
    assert h16.shape[0] == M
    # fp32 output: with these unnormalised synthetic magnitudes |y| reaches ~2.5e5,
    # beyond the fp16 range.
    y = q.jllm_q4k_gemm(dev(weights["down"]), dev(h16), H, F, out_dtype=torch.float32).cpu().numpy()
    if cols is None:
        ref, s = oracle.matmul(weights["down"], h16, H, F)
        assert_within(y, ref, s, f"down M={M}")
    else:
        dcols = sample_cols(H, rng, n_random=96)
        ref, s = oracle_matmul_rows(weights["down"], h16, H, F, cols=dcols)
        assert_within(y[:, dcols], ref, s, f"down M={M} (all rows, {len(dcols)} columns)")


@pytest.mark.parametrize("M", [1, 512])
def test_lm_head(q, M):
    import torch

    w = synthetic.q4k_weights(V, H, synthetic.weight_seed(4, 0, 7))
    x = synthetic.activations(M, H, synthetic.activation_seed(4, M, 7))
    y = q.jllm_q4k_gemm(dev(w), dev(x), V, H, out_dtype=torch.float32).cpu().numpy()
    if M == 1:
        ref, s = oracle.matmul(w, x, V, H)
        assert_within(y, ref, s, "lm head M=1")
    else:
        rng = np.random.Generator(np.random.PCG64(9))
        cols = sample_cols(V, rng, n_random=96)
        ref, s = oracle.matmul_cols(w, x, V, H, cols)
        assert_within(y[:, cols], ref, s, "lm head M=512")

"""Fused SwiGLU of the tcgen05 GEMM: h = silu(X Wg^T) * (X Wu^T) in fp16.

A tile's 128 rows pair 64 gate rows with the 64 up rows of the same outputs
(in each 32-lane quarter of tensor memory, lanes 0-15 gate and 16-31 up), so
the launch takes the plain tile shapes: tensor-memory A for up to 128 tokens,
256-token tiles (two accumulators, so that the exchange and silu of the
epilogue overlap the next tile), and the stream-K split.
The cases cover output widths that are not a multiple of 64 (a last pair tile
whose rows past N read as zero and are not stored), each tile shape, split and
whole tiles, and the full-size gate/up at M = 2048 (sampled columns, every
token).  Every checked element is within the oracle's SwiGLU bound."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import dev, oracle_matmul_rows, sample_cols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def _check(h, wg, wu, x, N, K, cols, label):
    g, sg = oracle_matmul_rows(wg, x, N, K, cols)
    u, su = oracle_matmul_rows(wu, x, N, K, cols)
    ref = oracle.swiglu(g, u)
    tol = oracle.swiglu_tolerance(g, u, sg, su)
    got = h[:, cols].astype(np.float64)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{label}: {int(bad.sum())} of {bad.size} outside the bound"


# (N, K, M)
CASES = [
    (100, 512, 5),       # one full and one 36-column pair tile, 16 tokens (A in tensor memory)
    (200, 768, 33),
    (1000, 2560, 129),   # 144-token tiles
    (640, 1024, 256),    # one 256-token tile
    (1000, 1280, 300),   # two token tiles (256 + 44)
]


@pytest.mark.parametrize("N,K,M", CASES)
def test_swiglu_pairs(q, N, K, M):
    import torch

    wg = synthetic.q4k_weights(N, K, 6100 + N)
    wu = synthetic.q4k_weights(N, K, 6200 + N)
    x = synthetic.activations(M, K, 6300 + M, per_token_scale=True)
    wgd, wud, xd = dev(wg), dev(wu), dev(x)
    h_split = q.jllm_q4k_ffn_swiglu(wgd, wud, xd, N, K, ws=q.workspace(M, N, K))
    h_whole = q.jllm_q4k_ffn_swiglu(wgd, wud, xd, N, K, ws=False)
    assert h_split.dtype == torch.float16 and h_split.shape == (M, N)
    cols = np.arange(N, dtype=np.int64)
    _check(h_split.float().cpu().numpy(), wg, wu, x, N, K, cols, f"split N={N} K={K} M={M}")
    _check(h_whole.float().cpu().numpy(), wg, wu, x, N, K, cols, f"whole N={N} K={K} M={M}")
    assert q.jllm_get_device_error() == 0


def test_swiglu_pairs_full_size(q):
    """gate/up 2560 -> 9728 at M = 2048: 152 pair tiles x 8 token tiles of 256."""
    N, K, M = 9728, 2560, 2048
    wg = synthetic.q4k_weights(N, K, synthetic.weight_seed(4, 0, 4))
    wu = synthetic.q4k_weights(N, K, synthetic.weight_seed(4, 0, 5))
    x = synthetic.activations(M, K, 6400)
    h = q.jllm_q4k_ffn_swiglu(dev(wg), dev(wu), dev(x), N, K).float().cpu().numpy()
    rng = np.random.Generator(np.random.PCG64(6401))
    cols = sample_cols(N, rng, n_random=40, edge=16, tile=64)
    _check(h, wg, wu, x, N, K, cols, "M=2048")
    assert np.all(np.isfinite(h))
    assert q.jllm_get_device_error() == 0

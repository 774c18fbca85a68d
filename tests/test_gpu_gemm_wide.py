"""Wide tiles of the tcgen05 GEMM (more than 256 tokens per tile, two MMAs of
half the tile per K slice into one 512-column accumulator).

The launch takes them when M > 256 and there are at least as many wide tiles as
SMs, so the shapes here have >= 152 weight-row tiles (N >= 19456) and a small K.
The token counts cover what the wide path splits differently: one tile of 320,
384 or 512 tokens (halves of 160, 192, 256), a second half cut short by M (449,
511), two and three token tiles (600, 1025), a ragged last weight-row tile, a
stream-K split of wide tiles (tile count not a multiple of the SM count), fp32
and fp16 output, and a batched launch.  Every token row of sampled columns is
compared with the oracle (the columns cover the first and last tiles, the
ragged tail and random tiles)."""
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


def _sms():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


def _check(y, w, x, N, K, cols, f16, label):
    ref, s = oracle_matmul_rows(w, x, N, K, cols)
    got = y[:, cols]
    tol = oracle.tolerance(s) + (2.0**-11 * np.abs(ref) + 2.0**-24 if f16 else 0.0)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{label}: {int(bad.sum())} of {bad.size} outside the bound"
    assert np.all(np.isfinite(y)), label


# (N, K, M, fp16 out)
CASES = [
    (19456, 256, 257, False),   # 152 row tiles x one tile of 320 tokens
    (19456, 512, 449, True),    # one tile of 512, the second half 193 tokens
    (19520, 768, 511, False),   # ragged last row tile; 512 tokens, 255 in half 1
    (19584, 256, 600, True),    # 153 x 2 tiles of 320: not a multiple of the SMs (split)
    (19456, 256, 1025, False),  # three tiles of 384
]


@pytest.mark.parametrize("N,K,M,f16", CASES)
def test_wide_tiles(q, N, K, M, f16):
    import torch

    if (N + 127) // 128 < _sms():
        pytest.skip("fewer weight-row tiles than SMs on this device")
    w = synthetic.q4k_weights(N, K, 4100 + M)
    x = synthetic.activations(M, K, 4200 + M, per_token_scale=True)
    wd, xd = dev(w), dev(x)
    dt = torch.float16 if f16 else torch.float32
    y = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt)
    y_again = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt)
    assert torch.equal(y, y_again)  # deterministic, also with the split
    y_whole = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt, ws=False)
    rng = np.random.Generator(np.random.PCG64(M))
    cols = sample_cols(N, rng, n_random=48, edge=16)
    label = f"N={N} K={K} M={M} f16={f16}"
    _check(y.float().cpu().numpy(), w, x, N, K, cols, f16, label + " split")
    _check(y_whole.float().cpu().numpy(), w, x, N, K, cols, f16, label + " whole")
    assert q.jllm_get_device_error() == 0


def test_wide_tiles_batched(q):
    """gate/up-style batch: two matrices of 9728 rows (152 row tiles together) on 300 tokens."""
    import torch

    Ns, K, M = [9728, 9728], 256, 300
    ws_np = [synthetic.q4k_weights(n, K, 4300 + i) for i, n in enumerate(Ns)]
    x = synthetic.activations(M, K, 4400, per_token_scale=True)
    ys = q.jllm_q4k_gemm_batch([dev(w) for w in ws_np], dev(x), Ns, K, out_dtype=torch.float16)
    rng = np.random.Generator(np.random.PCG64(7))
    for i, (w, n, y) in enumerate(zip(ws_np, Ns, ys)):
        cols = sample_cols(n, rng, n_random=32, edge=8)
        _check(y.float().cpu().numpy(), w, x, n, K, cols, True, f"batch matrix {i}")
    assert q.jllm_get_device_error() == 0

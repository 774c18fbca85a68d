"""The few-token GEMM (2 <= M <= 40): warp-level tensor cores on weights dequantised
in registers, K split over a thread-block cluster.

Each CTA takes 128 weight rows and T = 8 * ceil(M / 8) tokens; the launch
splits K into s = min(8, super-blocks, about two CTAs per SM / tiles) ranges,
one per CTA of a cluster, and the cluster adds its partial sums in rank order.
jllm_q4k_gemm sends M <= 24, and M <= 40 when W has at most 64 tiles of 128
rows, to it (the cases below are all such calls); a child process with
JLLM_GEMM_MMA_MAX_M=40 also sends it the large shapes.  The cases cover every
token-tile size (T = 8 .. 40), a single row tile (s = 8), super-block counts
that s does not divide and that limit s (K = 256: s = 1), ragged last row
tiles and odd N (element stores), fp32 and fp16 output, batches whose tiles
span matrices, the layer shapes at M = 33 as dispatched, closed-form edge rows
with mixed-magnitude activations, unit vectors, and determinism.  Every
compared element is within the oracle's matmul bound."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synthetic
from edge_inputs import N_KINDS, edge_weights, mixed_activations
from gpu_helpers import LAYER_SHAPES, assert_within, dev, oracle_matmul_rows, sample_cols

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    if bit_q4_weight_gb300.jllm_q4k_gemv_max_m() >= 2:
        pytest.skip("a few tokens run the CUDA-core GEMV under this threshold")
    if os.environ.get("JLLM_GEMM_MMA_MAX_M") is not None:
        pytest.skip("the dispatch rule is overridden in this process")
    return bit_q4_weight_gb300


def _f16_tol(ref, s):
    return oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24


# (N, K, M)
CASES = [
    (1000, 2560, 2),     # 8 tiles, T = 8 (2 of 8 tokens), s = 8
    (130, 4096, 4),      # 2 tiles (the second 2 rows), s = 8 over 16 super-blocks
    (128, 2560, 5),      # one tile, T = 8, s = 8 over 10 super-blocks
    (100, 512, 8),       # one partial tile, 2 super-blocks: s = 2
    (300, 256, 16),      # 3 tiles, K = 256: no split
    (1001, 4096, 17),    # 8 tiles (the last ragged, N odd: element stores), T = 24
    (4096, 2560, 23),    # 32 tiles (M <= 24 takes any shape), s = 9 -> 8
    (200, 2560, 24),     # T = 24, 2 tiles
    (520, 1280, 26),     # T = 32, 5 super-blocks: s = 5
    (640, 768, 32),      # T = 32, 3 super-blocks: s = 3
    (2560, 9728, 33),    # the down projection: 20 tiles, s = 8 over 38 super-blocks, T = 40
    (3072, 2560, 40),    # 24 tiles, T = 40
    (8064, 2560, 37),    # 63 tiles, T = 40
]


@pytest.mark.parametrize("N,K,M", CASES)
@pytest.mark.parametrize("f16", [False, True])
def test_few_token_gemm(q, N, K, M, f16):
    import torch

    w = synthetic.q4k_weights(N, K, 7100 + N + M)
    x = synthetic.activations(M, K, 7200 + M, per_token_scale=True)
    ref, s = oracle_matmul_rows(w, x, N, K)
    wd, xd = dev(w), dev(x)
    dt = torch.float16 if f16 else torch.float32
    y = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt)
    assert torch.equal(y, q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt))  # deterministic
    assert torch.equal(y, q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt, ws=False))  # no workspace used
    got = y.float().cpu().numpy()
    if f16:
        bad = np.abs(got - ref) > _f16_tol(ref, s)
        assert not bad.any(), f"N={N} K={K} M={M} fp16: {int(bad.sum())} outside"
    else:
        assert_within(got, ref, s, f"N={N} K={K} M={M}")
    assert q.jllm_get_device_error() == 0


@pytest.mark.parametrize("M", [9, 24, 40])
def test_few_token_gemm_batch(q, M):
    """Three matrices over one x (tiles of one launch span the matrices, ragged ends)."""
    import torch

    Ns, K = [1000, 600, 840], 2560
    ws_np = [synthetic.q4k_weights(n, K, 7300 + i) for i, n in enumerate(Ns)]
    x = synthetic.activations(M, K, 7400 + M, per_token_scale=True)
    wd = [dev(w) for w in ws_np]
    ys = q.jllm_q4k_gemm_batch(wd, dev(x), Ns, K, out_dtype=torch.float32)
    for i, (w, n) in enumerate(zip(ws_np, Ns)):
        ref, s = oracle.matmul(w, x, n, K)
        assert_within(ys[i].cpu().numpy(), ref, s, f"batch[{i}] M={M}")
    assert q.jllm_get_device_error() == 0


@pytest.mark.parametrize("M", [8, 16, 33])
def test_few_token_gemm_layer_shapes(q, M):
    """q/k/v and gate/up batches and o, down of the layer sweep, as the short-prefill
    bench launches them (at M = 33 the gate/up batch takes the tcgen05 kernel), fp16
    out: every token of sampled columns."""
    import torch

    rng = np.random.Generator(np.random.PCG64(M))
    shapes = {name: (K, N, idx) for idx, (name, K, N) in enumerate(LAYER_SHAPES)}
    for group in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)):
        K = shapes[group[0]][0]
        Ns = [shapes[g][1] for g in group]
        ws_np = [synthetic.q4k_weights(shapes[g][1], K, synthetic.weight_seed(7, 0, shapes[g][2])) for g in group]
        x = synthetic.activations(M, K, synthetic.activation_seed(7, M, K))
        ys = q.jllm_q4k_gemm_batch([dev(w) for w in ws_np], dev(x), Ns, K, out_dtype=torch.float16)
        for i, (w, n) in enumerate(zip(ws_np, Ns)):
            cols = sample_cols(n, rng, n_random=48, edge=16)
            ref, s = oracle_matmul_rows(w, x, n, K, cols)
            got = ys[i].float().cpu().numpy()[:, cols]
            bad = np.abs(got - ref) > _f16_tol(ref, s)
            assert not bad.any(), f"{group[i]}: {int(bad.sum())} outside"
    assert q.jllm_get_device_error() == 0


@pytest.mark.parametrize("M,K", [(33, 2560), (13, 9728), (40, 1280)])
def test_few_token_gemm_edge_rows(q, M, K):
    """Closed-form rows (zero rows, codes 15, large and subnormal d / dmin, min-only
    rows) against mixed-magnitude activations; the rows that are exactly zero give 0."""
    import torch

    N = 640
    w = edge_weights(N, K, 7500 + M)
    x = mixed_activations(M, K, 7600 + M)
    ref, s = oracle_matmul_rows(w, x, N, K)
    y = q.jllm_q4k_gemm(dev(w), dev(x), N, K, out_dtype=torch.float32).cpu().numpy()
    assert_within(y, ref, s, f"edge rows M={M} K={K}")
    zero = [n for n in range(N) if n % N_KINDS in (1, 3)]
    assert np.all(y[:, zero] == 0.0)
    assert q.jllm_get_device_error() == 0


def test_few_token_gemm_unit_vectors(q):
    """x rows = unit vectors: y = the weight itself, d*sc*q - dmin*m, up to fp32
    rounding of its two terms (the factored form: the code product is exact, the min
    term an exact fp16 hi + lo pair, fp32 sums): |y - w| <= 2^-22 (|w| + 2 dmin m),
    w and dmin*m exact from the oracle's block decode."""
    import torch

    N, K = 130, 512
    w = synthetic.q4k_weights(N, K, 1400)
    ks = np.array([0, 1, 2, 31, 32, 33, 63, 64, 100, 127, 128, 200, 255, 256, 300, 511])
    x = np.zeros((len(ks), K), dtype=np.float16)
    x[np.arange(len(ks)), ks] = 1.0
    y = q.jllm_q4k_gemm(dev(w), dev(x), N, K, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    blocks = w.reshape(N, K // 256, 144)
    for n in range(N):
        for i, k in enumerate(ks):
            blk = blocks[n, k // 256]
            exact = oracle.decode_block(blk)[k % 256]
            dmin = oracle.half_bits_to_double(blk[2:4].view(np.uint16))[0]
            _, m = oracle.scale_min(blk[4:16], (k % 256) // 32)
            bound = 2.0**-22 * (abs(exact) + 2 * abs(dmin * m))
            assert abs(y[i, n] - exact) <= bound, (n, k, y[i, n], exact)


CHILD = r"""
import sys
import numpy as np, torch
root = sys.argv[1]
sys.path.insert(0, root); sys.path.insert(0, root + "/tests")
import oracle, synthetic
from gpu_helpers import oracle_matmul_rows, sample_cols
import bit_q4_weight_gb300 as q
rng = np.random.Generator(np.random.PCG64(77))
# shapes the default rule sends to the tcgen05 kernel: many row tiles at 25..40 tokens
for Ns, K, M in (([4096, 4096, 1024], 2560, 33), ([9728, 9728], 2560, 40), ([19456], 512, 25)):
    ws_np = [synthetic.q4k_weights(n, K, 7700 + i + M) for i, n in enumerate(Ns)]
    x = synthetic.activations(M, K, 7800 + M, per_token_scale=True)
    ys = q.jllm_q4k_gemm_batch([torch.from_numpy(w).cuda() for w in ws_np], torch.from_numpy(x).cuda(), Ns, K,
                               out_dtype=torch.float32)
    for i, (w, n) in enumerate(zip(ws_np, Ns)):
        cols = sample_cols(n, rng, n_random=48, edge=16)
        ref, s = oracle_matmul_rows(w, x, n, K, cols)
        got = ys[i].cpu().numpy()[:, cols].astype(np.float64)
        assert np.all(np.abs(got - ref) <= oracle.tolerance(s)), (Ns, M, i)
assert q.jllm_get_device_error() == 0
print("ok")
"""


def test_few_token_gemm_forced_on_large_shapes():
    """JLLM_GEMM_MMA_MAX_M=40: batches of 72 and 152 row tiles at 33 and 40 tokens and
    152 row tiles at 25 tokens through the few-token kernel (child process)."""
    env = dict(os.environ, JLLM_GEMM_MMA_MAX_M="40")
    out = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stderr[-3000:]

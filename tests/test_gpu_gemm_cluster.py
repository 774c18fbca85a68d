"""Cluster split-K of the tcgen05 GEMM (tiles of at most 128 tokens that do not
fill the SMs): a cluster of s CTAs per tile, each taking 1/s of the tile's K
steps, the fp32 partials added in K order through distributed shared memory.

The shapes choose different cluster sizes through the tile count and the K
steps (s = min(8, SMs / tiles, K steps), lowered until the clusters fit at once;
below 4 the launch keeps the stream-K split):
K steps that s does not divide, s limited by a short K, one tile, ragged weight
rows and token tails, fp32 and fp16 output, and a batch whose tiles span
matrices.  Every element is compared with the oracle; the result does not depend
on whether a workspace is passed (the path uses none) and repeats bit for bit.
By default 5..40 tokens on few row tiles take the few-token GEMM, so these cases
use 41..128 tokens; a child process with JLLM_GEMM_MMA_MAX_M=0 runs the split at
5..33 tokens as well."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_within, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


# (N, K, M): tiles = ceil(N / 128), K steps = K / 128; s = min(8, SMs / tiles,
# K steps) when that is at least 4 (on 152 SMs)
# (M above 40: fewer tokens with these few row tiles take the few-token GEMM)
CASES = [
    (128, 512, 41),     # one tile, 4 K steps: s = 4, one step per CTA
    (200, 1792, 48),    # 2 tiles, 14 K steps: s = 8, steps 1-2 per CTA
    (1000, 2816, 50),   # 8 tiles (the last ragged), 22 K steps: s = 8
    (2560, 9728, 64),   # 20 tiles, 76 K steps: s = 7, the down projection at M = 64
    (4096, 2560, 100),  # 32 tiles, 20 K steps: s = 4
    (300, 768, 128),    # 3 tiles, 6 K steps: s = 6; a full 128-token tile
    (520, 1280, 45),    # 5 tiles, 10 K steps: s = 8, K steps not a multiple of s
]


@pytest.mark.parametrize("N,K,M", CASES)
@pytest.mark.parametrize("f16", [False, True])
def test_cluster_split(q, N, K, M, f16):
    import torch

    w = synthetic.q4k_weights(N, K, 5100 + N)
    x = synthetic.activations(M, K, 5200 + M, per_token_scale=True)
    ref, s = oracle.matmul(w, x, N, K)
    wd, xd = dev(w), dev(x)
    dt = torch.float16 if f16 else torch.float32
    y = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt)
    y_nows = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt, ws=False)
    assert torch.equal(y, y_nows)
    assert torch.equal(y, q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=dt))
    got = y.float().cpu().numpy()
    if f16:
        tol = oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24
        bad = np.abs(got - ref) > tol
        assert not bad.any(), f"N={N} K={K} M={M} fp16: {int(bad.sum())} outside"
    else:
        assert_within(got, ref, s, f"N={N} K={K} M={M}")
    assert q.jllm_get_device_error() == 0


def test_cluster_split_batch(q):
    """A batch of three matrices at M = 56: 8 + 5 + 7 = 20 tiles, s = 7, the last
    tile of each matrix ragged."""
    import torch

    Ns, K, M = [1000, 600, 840], 2560, 56
    ws_np = [synthetic.q4k_weights(n, K, 5300 + i) for i, n in enumerate(Ns)]
    x = synthetic.activations(M, K, 5400, per_token_scale=True)
    ys = q.jllm_q4k_gemm_batch([dev(w) for w in ws_np], dev(x), Ns, K, out_dtype=torch.float32)
    for i, (w, n, y) in enumerate(zip(ws_np, Ns, ys)):
        ref, s = oracle.matmul(w, x, n, K)
        assert_within(y.cpu().numpy(), ref, s, f"batch matrix {i}")
    assert q.jllm_get_device_error() == 0


CHILD = r"""
import sys
import numpy as np, torch
root = sys.argv[1]
sys.path.insert(0, root); sys.path.insert(0, root + "/tests")
import oracle, synthetic
import bit_q4_weight_gb300 as q
# the tcgen05 GEMM at the few-token sizes (the cluster split for narrow tiles, A in
# tensor memory), as JLLM_GEMM_MMA_MAX_M=0 selects it
for N, K, M in ((128, 512, 16), (200, 1792, 33), (2560, 9728, 33), (520, 1280, 20), (1000, 2560, 5)):
    w = synthetic.q4k_weights(N, K, 5700 + N + M)
    x = synthetic.activations(M, K, 5800 + M, per_token_scale=True)
    ref, s = oracle.matmul(w, x, N, K)
    wd, xd = torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda()
    y = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=torch.float32)
    assert torch.equal(y, q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=torch.float32, ws=False)), (N, K, M)
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - ref) <= oracle.tolerance(s)), (N, K, M)
assert q.jllm_get_device_error() == 0
print("ok")
"""


def test_cluster_split_at_few_tokens_when_selected():
    """JLLM_GEMM_MMA_MAX_M=0 keeps the tcgen05 GEMM for 5..40 tokens: its cluster split
    and narrow tiles there (child process: the variable is read once per process)."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, JLLM_GEMM_MMA_MAX_M="0")
    out = subprocess.run([sys.executable, "-c", CHILD, root], env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stderr[-3000:]

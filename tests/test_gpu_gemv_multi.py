"""CUDA-core GEMV for a few tokens (M = 2..8) through jllm_q4k_gemm.

The C ABI sends only M = 1 to the GEMV by default: from two tokens the
few-token tensor-core GEMM is faster on every layer shape.  JLLM_GEMV_MAX_M
(read once per process) raises the threshold, so the multi-token cases run in a
child process with it at 8: every M = 2..8 on three shapes, fp16 output, rows
that match the single-token GEMV, and closed-form edge rows with
mixed-magnitude activations (the rows that are exactly zero give 0)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def test_default_threshold_is_one_token(q):
    if os.environ.get("JLLM_GEMV_MAX_M") is not None:
        pytest.skip("the threshold is overridden in this process")
    assert q.jllm_q4k_gemv_max_m() == 1
    assert q.jllm_q4k_workspace_bytes(1, 1024, 2560) == 0  # the GEMV takes none


CHILD = r'''
import sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import bit_q4_weight_gb300 as q, oracle, synthetic
from edge_inputs import edge_weights, mixed_activations, CAP_FINITE
assert q.jllm_q4k_gemv_max_m() == 8
dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
for M in range(2, 9):
    for N, K in ((300, 2560), (1000, 9728), (129, 512)):
        w = synthetic.q4k_weights(N, K, 5000 + N + M)
        x = synthetic.activations(M, K, 5100 + M, per_token_scale=True)
        ref, s = oracle.matmul(w, x, N, K)
        y = q.jllm_q4k_gemm(dev(w), dev(x), N, K, out_dtype=torch.float32).cpu().numpy()
        assert np.all(np.abs(y - ref) <= oracle.tolerance(s)), ("fp32", M, N, K)
for M in (2, 4, 8):
    N, K = 512, 4096
    w = synthetic.q4k_weights(N, K, 5200 + M); x = synthetic.activations(M, K, 5300 + M)
    ref, s = oracle.matmul(w, x, N, K)
    y = q.jllm_q4k_gemm(dev(w), dev(x), N, K, out_dtype=torch.float16).float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y - ref) <= oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24), ("fp16", M)
# the rows of a multi-token call against single-token calls
N, K, M = 640, 2560, 6
w = synthetic.q4k_weights(N, K, 5400); x = synthetic.activations(M, K, 5401)
ref, s = oracle.matmul(w, x, N, K)
wd = dev(w)
y = q.jllm_q4k_gemm(wd, dev(x), N, K).cpu().numpy()
for m in range(M):
    g = q.jllm_q4k_gemv(wd, dev(x[m]), N, K).cpu().numpy()
    assert np.all(np.abs(g - y[m]) <= 2 * oracle.tolerance(s[m])), ("rows", m)
# closed-form edge rows, any finite d / dmin
for M, N, K in ((2, 384, 2560), (3, 384, 2560), (4, 384, 2560), (5, 256, 2560), (8, 200, 9728)):
    w = edge_weights(N, K, 7600 + M, cap_bits=CAP_FINITE); x = mixed_activations(M, K, 7700 + M)
    ref, s = oracle.matmul(w, x, N, K)
    y = q.jllm_q4k_gemm(dev(w), dev(x), N, K).cpu().numpy()
    assert np.all(np.abs(y - ref) <= oracle.tolerance(s)), ("edge", M, N, K)
    z = [n for n in range(N) if n % 8 in (1, 3)]
    assert np.all(y[:, z] == 0.0)
assert q.jllm_get_device_error() == 0
print("ok")
'''


def test_multi_token_gemv_through_threshold_override():
    env = dict(os.environ, JLLM_GEMV_MAX_M="8")
    out = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stderr[-3000:]

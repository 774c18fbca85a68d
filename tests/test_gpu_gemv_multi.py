"""CUDA-core GEMV for a few tokens (M = 2..jllm_q4k_gemv_max_m()) through jllm_q4k_gemm."""
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


def test_threshold_covers_small_m(q):
    assert q.jllm_q4k_gemv_max_m() >= 2
    assert q.jllm_q4k_workspace_bytes(q.jllm_q4k_gemv_max_m(), 1024, 2560) == 0  # the GEMV takes none


@pytest.mark.parametrize("M", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(300, 2560), (1000, 9728), (129, 512)])
def test_multi_token_gemv_matches_oracle(q, M, N, K):
    import torch

    if M > q.jllm_q4k_gemv_max_m():
        pytest.skip("above the dispatch threshold")
    w = synthetic.q4k_weights(N, K, 5000 + N + M)
    x = synthetic.activations(M, K, 5100 + M, per_token_scale=True)
    ref, s = oracle.matmul(w, x, N, K)
    y = q.jllm_q4k_gemm(dev(w), dev(x), N, K, out_dtype=torch.float32)
    assert_within(y.cpu().numpy(), ref, s, f"M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [2, 4, 8])
def test_multi_token_fp16_output(q, M):
    import torch

    N, K = 512, 4096
    w = synthetic.q4k_weights(N, K, 5200 + M)
    x = synthetic.activations(M, K, 5300 + M)
    ref, s = oracle.matmul(w, x, N, K)
    y = q.jllm_q4k_gemm(dev(w), dev(x), N, K, out_dtype=torch.float16).float().cpu().numpy().astype(np.float64)
    tol = oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24
    assert np.all(np.abs(y - ref) <= tol)


def test_multi_token_rows_match_single_token(q):
    N, K, M = 640, 2560, 6
    w = synthetic.q4k_weights(N, K, 5400)
    x = synthetic.activations(M, K, 5401)
    ref, s = oracle.matmul(w, x, N, K)
    wd = dev(w)
    y = q.jllm_q4k_gemm(wd, dev(x), N, K).cpu().numpy()
    for m in range(M):
        g = q.jllm_q4k_gemv(wd, dev(x[m]), N, K).cpu().numpy()
        assert np.all(np.abs(g - y[m]) <= 2 * oracle.tolerance(s[m]))
    assert q.jllm_get_device_error() == 0


def test_eight_token_kernel_through_threshold_override(tmp_path):
    """M = 5..8 run the 8-token kernel when JLLM_GEMV_MAX_M raises the threshold (read once
    per process, so this runs in a child process)."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = r'''
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import bit_q4_weight_gb300 as q, oracle, synthetic
assert q.jllm_q4k_gemv_max_m() == 8
for M, N, K in ((7, 300, 2560), (8, 129, 9728), (5, 64, 512)):
    w = synthetic.q4k_weights(N, K, 5500 + M); x = synthetic.activations(M, K, 5600 + M)
    ref, s = oracle.matmul(w, x, N, K)
    y = q.jllm_q4k_gemm(torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda(), N, K).cpu().numpy()
    assert np.all(np.abs(y - ref) <= oracle.tolerance(s)), (M, N, K)
assert q.jllm_get_device_error() == 0
print("ok")
'''
    env = dict(os.environ, JLLM_GEMV_MAX_M="8")
    out = subprocess.run([sys.executable, "-c", code, root], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stderr[-2000:]

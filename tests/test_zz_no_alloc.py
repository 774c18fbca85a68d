"""jllm_q4k_gemm_noalloc: the stream-K GEMM on the library's static device
workspace.  Collected last (file name) so that it also runs after every other
test has used the library; it passes on its own as well."""
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


# cut tiles on the static array (stream-K: 20 tiles of 256 tokens, 64 K steps), whole
# tiles (64 of 20 steps), the cluster split (3 and 20 narrow tiles, a ragged tail),
# M = 33 on 8 row tiles (the few-token GEMM), and M at the GEMV threshold -- none but
# the first touches the array, and every one must leave it reusable
@pytest.mark.parametrize("N,K,M", [(1280, 4096, 300), (1024, 2560, 33), (4096, 2560, 235), (300, 1280, 70),
                                   (2560, 9728, 64), (256, 512, 1)])
def test_noalloc_matches_oracle_and_caller_workspace(q, N, K, M):
    import torch

    w = synthetic.q4k_weights(N, K, 3100 + N)
    x = synthetic.activations(M, K, 3200 + M, per_token_scale=True)
    ref, s = oracle.matmul(w, x, N, K)
    wd, xd = dev(w), dev(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y2 = torch.empty_like(y)
    q.jllm_q4k_gemm_noalloc(wd, xd, N, K, out=y)  # first use loads the module (and its static array)
    torch.cuda.synchronize()
    # Process-local counters (torch's allocator) and the device-wide free memory; the
    # latter assumes no other process allocates on this GPU meanwhile.
    before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
    q.jllm_q4k_gemm_noalloc(wd, xd, N, K, out=y)
    q.jllm_q4k_gemm_noalloc(wd, xd, N, K, out=y2)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
    assert after == before  # the calls allocate no device memory
    assert_within(y.cpu().numpy(), ref, s, f"noalloc N={N} K={K} M={M}")
    assert torch.equal(y, y2)  # the static workspace is left reusable
    # same split, same order of partial sums as a caller-provided workspace
    y_ws = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=torch.float32, ws=q.workspace(M, N, K))
    assert torch.equal(y, y_ws)
    assert q.jllm_get_device_error() == 0


def test_noalloc_fp16_and_argument_errors(q):
    import torch

    N, K, M = 1280, 4096, 256
    w = synthetic.q4k_weights(N, K, 3300)
    x = synthetic.activations(M, K, 3301)
    ref, s = oracle.matmul(w, x, N, K)
    y = q.jllm_q4k_gemm_noalloc(dev(w), dev(x), N, K, out_dtype=torch.float16).float().cpu().numpy()
    tol = oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24
    assert np.all(np.abs(y.astype(np.float64) - ref) <= tol)
    assert q.lib.jllm_q4k_gemm_noalloc(None, None, None, 0, M, N, K, None) == 1  # INVALID_ARG
    wd, xd = dev(w), dev(x)
    yd = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert q.lib.jllm_q4k_gemm_noalloc(wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), 0, M, N, K - 1, None) == 2

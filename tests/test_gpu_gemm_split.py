"""Stream-K split of the tcgen05 GEMM: cut tiles summed across CTAs through the
workspace must stay within the matmul bound of the oracle, be deterministic,
and leave the workspace reusable."""
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


def _sms():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


# (N, K, M): tile counts that do not fill the SMs evenly, so K ranges are cut
# between CTAs where that shortens the busiest CTA by 12 K steps or more -- a tile
# over several CTAs (few tiles), ragged M and N tails.  Cut tiles of at most 128
# tokens (A in tensor memory): (6144, 4096, 64) with 48 tiles of 32 steps and
# (2560, 9728, 235) with 40 of 76 (the M = 235 down projection); of 129..256
# tokens: (300, 1280, 300), (1280, 4096, 600), (520, 2816, 1025).  (4096, 2560,
# 235) keeps whole tiles with a workspace (64 tiles of 20 steps); (1280, 4096,
# 256) and (200, 768, 70) take the cluster split.
SHAPES = [(6144, 4096, 64), (1280, 4096, 256), (200, 768, 70), (2560, 9728, 235), (300, 1280, 300), (4096, 2560, 235),
          (1280, 4096, 600), (520, 2816, 1025)]


@pytest.mark.parametrize("N,K,M", SHAPES)
def test_split_matches_oracle_and_whole_tiles(q, N, K, M):
    import torch

    w = synthetic.q4k_weights(N, K, 2100 + N)
    x = synthetic.activations(M, K, 2200 + M, per_token_scale=True)
    ref, s = oracle.matmul(w, x, N, K)
    wd, xd = dev(w), dev(x)
    ws = q.workspace(M, N, K)
    assert ws is not None and ws.numel() == q.jllm_q4k_workspace_bytes(M, N, K)
    y_split = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=torch.float32, ws=ws)
    y_whole = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=torch.float32, ws=False)
    assert_within(y_split.cpu().numpy(), ref, s, f"split N={N} K={K} M={M}")
    assert_within(y_whole.cpu().numpy(), ref, s, f"whole N={N} K={K} M={M}")
    # the two differ only by the order of fp32 partial sums
    assert np.all(np.abs(y_split.cpu().numpy() - y_whole.cpu().numpy()) <= 2 * oracle.tolerance(s))
    # deterministic: the same call again gives the same bits
    y_again = q.jllm_q4k_gemm(wd, xd, N, K, out_dtype=torch.float32, ws=ws)
    assert torch.equal(y_split, y_again)
    # the flag words (after one 256 KiB slot per SM) are back to zero
    sms = _sms()
    flags = ws[sms * 262144: sms * 262144 + 4 * sms]
    assert int(flags.count_nonzero()) == 0
    assert q.jllm_get_device_error() == 0


@pytest.mark.parametrize("M", [24, 100, 512])
def test_split_swiglu(q, M):
    import torch

    N, K = 1024, 2560
    wg = synthetic.q4k_weights(N, K, 2300)
    wu = synthetic.q4k_weights(N, K, 2301)
    x = synthetic.activations(M, K, 2302 + M)
    g, sg = oracle.matmul(wg, x, N, K)
    u, su = oracle.matmul(wu, x, N, K)
    ref = oracle.swiglu(g, u)
    tol = oracle.swiglu_tolerance(g, u, sg, su)
    ws = q.workspace(M, N, K)
    h = q.jllm_q4k_ffn_swiglu(dev(wg), dev(wu), dev(x), N, K, ws=ws).float().cpu().numpy()
    assert np.all(np.abs(h - ref) <= tol)
    h2 = q.jllm_q4k_ffn_swiglu(dev(wg), dev(wu), dev(x), N, K, ws=ws).float().cpu().numpy()
    assert np.array_equal(h, h2)
    sms = _sms()
    assert int(ws[sms * 262144: sms * 262144 + 4 * sms].count_nonzero()) == 0


def test_split_fp16_output(q):
    import torch

    N, K, M = 1024, 2560, 96
    w = synthetic.q4k_weights(N, K, 2400)
    x = synthetic.activations(M, K, 2401)
    ref, s = oracle.matmul(w, x, N, K)
    y = q.jllm_q4k_gemm(dev(w), dev(x), N, K, out_dtype=torch.float16, ws=q.workspace(M, N, K))
    y = y.float().cpu().numpy().astype(np.float64)
    tol = oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24
    assert np.all(np.abs(y - ref) <= tol)


def test_workspace_errors(q):
    import torch

    N, K, M = 256, 512, 64
    w = dev(synthetic.q4k_weights(N, K, 2500))
    x = dev(synthetic.activations(M, K, 2501))
    need = q.jllm_q4k_workspace_bytes(M, N, K)
    assert need > 0 and need % 256 == 0
    assert q.jllm_q4k_workspace_bytes(1, N, K) == 0  # the GEMV takes none
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.JllmError) as e:
        q.jllm_q4k_gemm(w, x, N, K, ws=small)
    assert "WORKSPACE" in str(e.value)
    big = torch.zeros(need + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.JllmError) as e:
        q.jllm_q4k_gemm(w, x, N, K, ws=big[16:])  # not 256-byte aligned
    assert "WORKSPACE" in str(e.value)

"""Producer -> consumer chains on one stream, enqueued back to back with no host
synchronisation: the consumer kernel is launched with programmatic dependent
launch and starts while its producer still runs, so these tests check that every
kernel reads its input only after the producer has finished.  The intermediate
buffer is filled with NaN before the chain, so an early read shows as NaN.

Expected values come from the oracle alone: the oracle's own intermediate
(h_ref) and the bound for a consumer whose input differs from h_ref by at most
the producer's own tolerance (gpu_helpers.chained_bound)."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import chained_bound, dev, oracle_matmul_rows

pytestmark = pytest.mark.gpu

H, F = 2560, 9728


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


@pytest.fixture(scope="module")
def ffn():
    return (synthetic.q4k_weights(F, H, synthetic.weight_seed(4, 1, 4)),
            synthetic.q4k_weights(F, H, synthetic.weight_seed(4, 1, 5)),
            synthetic.q4k_weights(H, F, synthetic.weight_seed(4, 1, 6)))


def _assert_bound(y, ref, bound, label):
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y)), f"{label}: non-finite outputs (input read before it was written?)"
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), f"{label}: {int(bad.sum())} outside the chained bound, worst excess {(err - bound).max():.3e}"


@pytest.mark.parametrize("M", [1, 512])
def test_swiglu_then_down_chain(q, ffn, M):
    """h = silu(x Wg^T) * (x Wu^T) (fp16) and y = h Wd^T (fp32), back to back."""
    import torch

    wg, wu, wd = ffn
    x = synthetic.activations(M, H, synthetic.activation_seed(4, M, 3))
    wgd, wud, wdd, xd = dev(wg), dev(wu), dev(wd), dev(x)
    h = torch.full((M, F), float("nan"), dtype=torch.float16, device="cuda")
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    for _ in range(3):  # repeated: later rounds find h already holding a previous result
        h.fill_(float("nan"))
        q.jllm_q4k_ffn_swiglu(wgd, wud, xd, F, H, out=h)
        q.jllm_q4k_gemm(wdd, h, H, F, out=y)
    torch.cuda.synchronize()
    rows = np.arange(M) if M == 1 else np.unique(np.r_[0:8, M - 8:M, np.random.Generator(
        np.random.PCG64(5)).integers(0, M, 48)])
    xr = x[rows]
    g, sg = oracle_matmul_rows(wg, xr, F, H)
    u, su = oracle_matmul_rows(wu, xr, F, H)
    h_ref = oracle.swiglu(g, u)
    t = oracle.swiglu_tolerance(g, u, sg, su)
    y_ref, _ = oracle_matmul_rows(wd, h_ref, H, F)
    bound = chained_bound(wd, h_ref, t, H, F)
    _assert_bound(y.cpu().numpy()[rows], y_ref, bound, f"swiglu->down M={M}")
    assert q.jllm_get_device_error() == 0


@pytest.mark.parametrize("M", [1, 3, 235])
def test_gemm_fp16_output_feeds_next_gemm(q, M):
    """Y1 = X W1^T (fp16 out) then Y2 = Y1 W2^T: GEMV -> GEMV (M = 1), few-token ->
    few-token (M = 3) or tcgen05 -> tcgen05."""
    import torch

    K1, N1, N2 = 2560, 4096, 1024
    w1 = synthetic.q4k_weights(N1, K1, 8700 + M)
    w2 = synthetic.q4k_weights(N2, N1, 8800 + M)
    x = synthetic.activations(M, K1, 8900 + M)
    w1d, w2d, xd = dev(w1), dev(w2), dev(x)
    y1 = torch.empty((M, N1), dtype=torch.float16, device="cuda")
    y2 = torch.empty((M, N2), dtype=torch.float32, device="cuda")
    for _ in range(3):
        y1.fill_(float("nan"))
        q.jllm_q4k_gemm(w1d, xd, N1, K1, out=y1)
        q.jllm_q4k_gemm(w2d, y1, N2, N1, out=y2)
    torch.cuda.synchronize()
    r1, s1 = oracle_matmul_rows(w1, x, N1, K1)
    t1 = oracle.tolerance(s1) + 2.0**-11 * np.abs(r1) + 2.0**-24  # fp16 output of the producer
    r2, _ = oracle_matmul_rows(w2, r1, N2, N1)
    bound = chained_bound(w2, r1, t1, N2, N1)
    _assert_bound(y2.cpu().numpy(), r2, bound, f"gemm->gemm M={M}")
    assert q.jllm_get_device_error() == 0


def test_gemv_batch_reads_previous_gemm_output(q):
    """A batched decode GEMV (q/k/v-like) reading the fp16 output of the GEMV before it."""
    import torch

    K0, K = 4096, 2560
    w0 = synthetic.q4k_weights(K, K0, 9000)
    ws = [synthetic.q4k_weights(n, K, 9001 + i) for i, n in enumerate((4096, 1024, 1024))]
    x = synthetic.activations(1, K0, 9010)
    w0d, xd = dev(w0), dev(x)
    wds = [dev(w) for w in ws]
    hid = torch.empty((1, K), dtype=torch.float16, device="cuda")
    outs = [torch.empty(n, dtype=torch.float32, device="cuda") for n in (4096, 1024, 1024)]
    for _ in range(3):
        hid.fill_(float("nan"))
        q.jllm_q4k_gemm(w0d, xd, K, K0, out=hid)
        q.jllm_q4k_gemv_batch(wds, hid.view(K), [4096, 1024, 1024], K, outs=outs)
    torch.cuda.synchronize()
    r0, s0 = oracle.matmul(w0, x, K, K0)
    t0 = oracle.tolerance(s0) + 2.0**-11 * np.abs(r0) + 2.0**-24
    for i, (w, n) in enumerate(zip(ws, (4096, 1024, 1024))):
        ref, _ = oracle.matmul(w, r0, n, K)
        _assert_bound(outs[i].cpu().numpy()[None, :], ref, chained_bound(w, r0, t0, n, K), f"batch matrix {i}")

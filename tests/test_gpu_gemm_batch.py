"""Batched tcgen05 GEMM (several weight matrices sharing X in one launch):
every output within the matmul bound of the fp64 oracle, bit-identical to
single calls when tiles are whole, deterministic with the stream-K split,
and the workspace flags back at zero."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import LAYER_SHAPES, assert_within, dev, sample_cols, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def _sms():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


# (Ns, K, M): ragged N tails inside the batch, one matrix of a single
# partial tile, M with a ragged token tile, and four matrices.
CASES = [
    ([256, 128, 128], 512, 40),
    ([200, 72, 384], 768, 70),
    ([1024, 256, 256], 2560, 235),
    ([96, 1000, 130, 512], 1280, 300),
    ([128], 512, 17),
    ([200, 72, 384], 768, 600),  # tiles of more than 256 tokens (two of 320)
]


@pytest.mark.parametrize("Ns,K,M", CASES)
def test_batch_matches_oracle_and_single_calls(q, Ns, K, M):
    import torch

    ws_np = [synthetic.q4k_weights(n, K, 3100 + 7 * i + n) for i, n in enumerate(Ns)]
    x = synthetic.activations(M, K, 3200 + M, per_token_scale=True)
    wd, xd = [dev(w) for w in ws_np], dev(x)
    whole = q.jllm_q4k_gemm_batch(wd, xd, Ns, K, out_dtype=torch.float32, ws=False)
    ws = q.workspace(M, sum(Ns), K)
    split = q.jllm_q4k_gemm_batch(wd, xd, Ns, K, out_dtype=torch.float32, ws=ws)
    again = q.jllm_q4k_gemm_batch(wd, xd, Ns, K, out_dtype=torch.float32, ws=ws)
    for i, (w, n) in enumerate(zip(ws_np, Ns)):
        ref, s = oracle.matmul(w, x, n, K)
        assert_within(whole[i].cpu().numpy(), ref, s, f"whole batch[{i}] N={n} K={K} M={M}")
        assert_within(split[i].cpu().numpy(), ref, s, f"split batch[{i}] N={n} K={K} M={M}")
        # the same sums as a single call, up to the order of the fp32 partial sums
        # (narrow tiles that do not fill the SMs split K over a cluster, and how
        # far depends on the launch's tile count)
        single = q.jllm_q4k_gemm(wd[i], xd, n, K, out_dtype=torch.float32, ws=False)
        diff = np.abs(whole[i].cpu().numpy().astype(np.float64) - single.cpu().numpy())
        assert np.all(diff <= 2 * oracle.tolerance(s)), f"batch[{i}] differs from the single call"
        assert torch.equal(split[i], again[i]), f"batch[{i}] not deterministic"
    if ws is not None:
        sms = _sms()
        assert int(ws[sms * 262144: sms * 262144 + 4 * sms].count_nonzero()) == 0
    assert q.jllm_get_device_error() == 0


def test_batch_fp16_output(q):
    import torch

    Ns, K, M = [384, 128, 128], 1024, 96
    ws_np = [synthetic.q4k_weights(n, K, 3300 + i) for i, n in enumerate(Ns)]
    x = synthetic.activations(M, K, 3310)
    ys = q.jllm_q4k_gemm_batch([dev(w) for w in ws_np], dev(x), Ns, K, out_dtype=torch.float16)
    for i, (w, n) in enumerate(zip(ws_np, Ns)):
        assert ys[i].dtype == torch.float16
        ref, s = oracle.matmul(w, x, n, K)
        got = ys[i].float().cpu().numpy()
        assert np.all(np.abs(got - ref) <= oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24)


@pytest.mark.parametrize("M", [1])
def test_batch_at_or_below_threshold_runs_gemv(q, M):
    import torch

    if M > q.jllm_q4k_gemv_max_m():
        pytest.skip("above the GEMV threshold")
    Ns, K = [256, 128], 512
    ws_np = [synthetic.q4k_weights(n, K, 3400 + i) for i, n in enumerate(Ns)]
    x = synthetic.activations(M, K, 3410 + M)
    wd, xd = [dev(w) for w in ws_np], dev(x)
    ys = q.jllm_q4k_gemm_batch(wd, xd, Ns, K, out_dtype=torch.float32)
    for i, (w, n) in enumerate(zip(ws_np, Ns)):
        ref, s = oracle.matmul(w, x, n, K)
        assert_within(ys[i].cpu().numpy(), ref, s, f"gemv batch[{i}] M={M}")
        assert torch.equal(ys[i], q.jllm_q4k_gemm(wd[i], xd, n, K, out_dtype=torch.float32))


@pytest.mark.parametrize("M", [33, 235, 2048])
def test_batch_qkv_and_gate_up_layer_shapes(q, M):
    """q/k/v (2560 -> 4096, 1024, 1024) and gate/up (2560 -> 9728 x 2) batches and
    o (4096 -> 2560) and down (9728 -> 2560) of the layer sweep, as the prefill
    bench launches them, fp16 out, with the workspace: sampled outputs against the
    oracle.  At M = 235 the q/k/v batch keeps whole tiles while o and down cut
    them (stream-K)."""
    import torch

    shapes = {name: (K, N, idx) for idx, (name, K, N) in enumerate(LAYER_SHAPES)}
    for group in (("q", "k", "v"), ("gate", "up"), ("o",), ("down",)):
        K = shapes[group[0]][0]
        Ns = [shapes[g][1] for g in group]
        ws_np = [synthetic.q4k_weights(shapes[g][1], K, synthetic.weight_seed(3, 0, shapes[g][2])) for g in group]
        x = synthetic.activations(M, K, synthetic.activation_seed(3, M, K))
        ys = q.jllm_q4k_gemm_batch([dev(w) for w in ws_np], dev(x), Ns, K, out_dtype=torch.float16,
                                   ws=q.workspace(M, sum(Ns), K))
        rng = np.random.Generator(np.random.PCG64(M + len(group)))
        rows = sample_rows(M, rng)
        for i, (w, n) in enumerate(zip(ws_np, Ns)):
            cols = sample_cols(n, rng, n_random=48, edge=16)
            ref, s = oracle.matmul_cols(w, x[rows], n, K, cols)
            got = ys[i].float().cpu().numpy()[np.ix_(rows, cols)]
            tol = oracle.tolerance(s) + 2.0**-11 * np.abs(ref) + 2.0**-24
            assert np.all(np.abs(got - ref) <= tol), f"{group[i]} M={M}"
    assert q.jllm_get_device_error() == 0

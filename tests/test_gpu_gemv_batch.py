"""Batched decode GEMV (several matrices, one shared x, one launch) vs the oracle."""
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


@pytest.mark.parametrize(
    "Ns,K",
    [
        ((4096, 1024, 1024), 2560),   # q, k, v of the attention block
        ((9728, 9728), 2560),         # gate, up of the MLP
        ((100, 1, 257, 64, 3, 129, 31, 500), 512),  # eight matrices, ragged row counts
        ((2560,), 9728),              # a batch of one
        ((300, 77), 4096),
    ],
)
def test_gemv_batch_matches_oracle(q, Ns, K):
    x = synthetic.activations(1, K, 4000 + K)
    ws = [synthetic.q4k_weights(n, K, 4100 + 13 * i + n) for i, n in enumerate(Ns)]
    xd = dev(x.reshape(K))
    outs = q.jllm_q4k_gemv_batch([dev(w) for w in ws], xd, Ns, K)
    for i, (w, n) in enumerate(zip(ws, Ns)):
        ref, s = oracle.matmul(w, x, n, K)
        assert_within(outs[i].cpu().numpy()[None, :], ref, s, f"matrix {i} of {Ns}")
        single = q.jllm_q4k_gemv(dev(w), xd, n, K).cpu().numpy()
        assert np.all(np.abs(single - outs[i].cpu().numpy()) <= 2 * oracle.tolerance(s[0]))
    assert q.jllm_get_device_error() == 0


def test_gemv_batch_outputs_untouched_beyond_rows(q):
    import torch

    K = 512
    Ns = (5, 70)
    x = synthetic.activations(1, K, 4200)
    ws = [dev(synthetic.q4k_weights(n, K, 4300 + n)) for n in Ns]
    bufs = [torch.full((n + 8,), 7.0, dtype=torch.float32, device="cuda") for n in Ns]
    q.jllm_q4k_gemv_batch(ws, dev(x.reshape(K)), Ns, K, outs=[b[:n] for b, n in zip(bufs, Ns)])
    for b, n in zip(bufs, Ns):
        assert torch.all(b[n:] == 7.0)

"""Fused q/k/v decode GEMV with the rotary epilogue (jllm_q4k_gemv_qkv_rope) vs
the oracle: matmul, optional RMSNorm of x, optional per-head RMSNorm of q and
k, RoPE at a position, on the Qwen3-4B attention shapes (32 query heads, 8 KV
heads of 128, hidden 2560).

Bound: each projected value t within the matmul bound E of the oracle's exact
t; the per-head norm and the rotation propagate it (below, from oracle
quantities only), plus fp32 rounding of the norm factor, the products and the
cosine and sine."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import dev

pytestmark = pytest.mark.gpu

HQ, HKV, D, K = 32, 8, 128, 2560
BASE = 1.0e6
U = 2.0**-24


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


@pytest.fixture(scope="module")
def weights():
    return [synthetic.q4k_weights(n, K, synthetic.weight_seed(1, 3, i)) for i, n in enumerate((HQ * D, HKV * D, HKV * D))]


def _norm_bound(t, E, g, eps):
    """Per-head RMSNorm n = t g / sqrt(mean t^2 + eps) of exact t, and the bound on |n' - n| for an
    input t' with |t' - t| <= E (first order with a (1 - delta)^-1.5 margin, plus fp32 rounding)."""
    th, Eh = t.reshape(-1, D), E.reshape(-1, D)
    n = oracle.head_rmsnorm(t, g, eps).reshape(-1, D)
    ss = np.sum(th * th, axis=1, keepdims=True)
    ds = np.sum(2 * np.abs(th) * Eh + Eh * Eh, axis=1, keepdims=True) + 32 * U * (ss + np.sum(Eh * Eh, axis=1, keepdims=True))
    den = ss + D * eps
    delta = ds / den
    assert np.all(delta < 0.5)
    r = 1.0 / np.sqrt(den / D)
    dr = r * (0.5 * delta / (1 - delta) ** 1.5 + 4 * U)
    En = np.abs(g) * (Eh * (r + dr) + np.abs(th) * dr) + 3 * U * np.abs(n)
    return n.reshape(t.shape), En.reshape(t.shape)


def _rope_bound(a, E):
    """Bound for the rotation of values a (exact) given input errors E: per pair (j, j+64),
    |c| E_j + |s| E_j+64 <= E_j + E_j+64, plus fp32 rounding of c, s and the products."""
    ah, Eh = a.reshape(-1, D), E.reshape(-1, D)
    pair = Eh[:, :64] + Eh[:, 64:]
    mag = np.abs(ah[:, :64]) + np.abs(ah[:, 64:])
    b = pair + 4 * U * mag
    return np.concatenate([b, b], axis=1).reshape(a.shape)


def _reference(weights, x, gamma, eps, q_gamma, k_gamma, head_eps, pos):
    xn = x.astype(np.float64) if gamma is None else oracle.rmsnorm(x.astype(np.float64), gamma.astype(np.float64), eps)
    outs = []
    for i, (w, n) in enumerate(zip(weights, (HQ * D, HKV * D, HKV * D))):
        t, s = oracle.matmul(w, xn, n, K)
        t, E = t[0], oracle.tolerance(s[0])
        hg = (q_gamma, k_gamma, None)[i]
        if i < 2:
            if hg is not None:
                t, E = _norm_bound(t, E, hg.astype(np.float64), head_eps)
            E = _rope_bound(t, E)
            t = oracle.rope(t, pos, BASE)
        outs.append((t, E))
    return outs


@pytest.mark.parametrize("pos", [0, 1, 1000, 32767, 123457])
@pytest.mark.parametrize("variant", ["rope", "headnorm", "full"])
def test_qkv_rope_matches_oracle(q, weights, pos, variant):
    rng = np.random.Generator(np.random.PCG64(9100 + pos))
    x = synthetic.activations(1, K, 9200 + pos)[0]
    gamma = rng.uniform(0.25, 2.0, size=K).astype(np.float32) if variant == "full" else None
    qg = rng.uniform(0.5, 1.5, size=D).astype(np.float32) if variant != "rope" else None
    kg = rng.uniform(0.5, 1.5, size=D).astype(np.float32) if variant != "rope" else None
    got = q.jllm_q4k_gemv_qkv_rope([dev(w) for w in weights], dev(x), HQ, HKV, K, pos, BASE,
                                   gamma=None if gamma is None else dev(gamma), eps=1e-6,
                                   q_gamma=None if qg is None else dev(qg), k_gamma=None if kg is None else dev(kg),
                                   head_eps=1e-6)
    ref = _reference(weights, x, gamma, 1e-6, qg, kg, 1e-6, pos)
    for name, g, (r, E) in zip("qkv", got, ref):
        y = g.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(y)), name
        err = np.abs(y - r)
        assert np.all(err <= E), f"{variant} pos={pos} {name}: {int((err > E).sum())} outside, worst {(err - E).max():.3e}"
    assert q.jllm_get_device_error() == 0


def test_rope_at_position_zero_is_the_plain_projection(q, weights):
    """pos = 0, no norms: cos 0 = 1 and sin 0 = 0, so q, k, v equal the batched GEMV's outputs bit
    for bit (same launch configuration and per-row arithmetic, so this pins the row placement)."""
    x = dev(synthetic.activations(1, K, 9300)[0])
    wd = [dev(w) for w in weights]
    got = q.jllm_q4k_gemv_qkv_rope(wd, x, HQ, HKV, K, 0, BASE)
    plain = q.jllm_q4k_gemv_batch(wd, x, [HQ * D, HKV * D, HKV * D], K)
    for a, b in zip(got, plain):
        assert np.array_equal(a.cpu().numpy(), b.cpu().numpy())


def test_rope_argument_errors(q, weights):
    import torch

    wd = [dev(w) for w in weights]
    x = dev(synthetic.activations(1, K, 9301)[0])
    ys = [torch.empty(n, dtype=torch.float32, device="cuda") for n in (HQ * D, HKV * D, HKV * D)]
    import ctypes

    wp = (ctypes.c_void_p * 3)(*[w.data_ptr() for w in wd])
    yp = (ctypes.c_void_p * 3)(*[y.data_ptr() for y in ys])
    s = torch.cuda.current_stream().cuda_stream
    call = lambda **kw: q.lib.jllm_q4k_gemv_qkv_rope(
        wp, yp, kw.get("hq", HQ), kw.get("hkv", HKV), x.data_ptr(), kw.get("K", K), None, 1e-6, None, None,
        kw.get("heps", 1e-6), kw.get("pos", 5), kw.get("base", 1e6), s)
    assert call() == 0
    assert call(hq=0) == 1
    assert call(base=0.0) == 1
    assert call(base=float("inf")) == 1
    assert call(pos=1 << 40) == 1
    assert call(K=300) == 2
    torch.cuda.synchronize()

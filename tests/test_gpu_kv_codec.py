"""FP16 <-> INT8 KV codec on the GPU vs the oracle: codes, scales and decoded
values bit-exact (integer codes decided in the same precision on both sides:
power-of-two scalings are exact), the round-trip bound and the no-drift fixed
point, on ragged counts, every head size and the full 4096-token Qwen3-4B cache."""
import numpy as np
import pytest

import oracle
from gpu_helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def _vectors(n, dim, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    mag = 10.0 ** rng.uniform(-9, 4.5, size=(n, 1))
    v = np.clip(rng.standard_normal((n, dim)) * mag, -65504, 65504).astype(np.float16)
    v[::97] = 0.0                                     # zero vectors
    v[1::89, 0] = np.float16(65504.0)                 # saturating maxima
    v[2::83] = (rng.integers(-127, 128, size=v[2::83].shape) * 2.0**-24).astype(np.float16)  # subnormal only
    return v


@pytest.mark.parametrize("dim", [64, 128, 256])
@pytest.mark.parametrize("n", [1, 3, 1000, 4099])
def test_kv_codec_bit_exact(q, dim, n):
    v = _vectors(n, dim, 9600 + n + dim)
    codes, scales = q.jllm_kv_encode_i8(dev(v), head_dim=dim)
    rq, rs = oracle.kv_encode(v, dim)
    assert np.array_equal(codes.cpu().numpy(), rq)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), rs.view(np.uint16))
    out = q.jllm_kv_decode_i8(codes, scales, head_dim=dim).cpu().numpy()
    assert np.array_equal(out.view(np.uint16), oracle.kv_decode(rq, rs, dim).view(np.uint16))


def test_kv_codec_full_cache_properties(q):
    """Qwen3-4B cache, 4096 tokens: 36 layers x {K, V} x 8 heads x 128 (2,359,296 vectors).
    Sampled vectors bit-exact against the oracle; on every vector, the no-drift fixed point and
    the round-trip bound."""
    import torch

    n = 36 * 2 * 8 * 4096
    g = torch.Generator(device="cuda").manual_seed(9700)
    kv = (torch.randn((n, 128), device="cuda", generator=g) *
          torch.exp(torch.randn((n, 1), device="cuda", generator=g) * 2.0)).clamp(-65504, 65504).half()
    codes, scales = q.jllm_kv_encode_i8(kv)
    back = q.jllm_kv_decode_i8(codes, scales)
    codes2, scales2 = q.jllm_kv_encode_i8(back)
    assert torch.equal(codes2, codes) and torch.equal(scales2, scales)
    assert torch.equal(q.jllm_kv_decode_i8(codes2, scales2), back)
    err = (back.float() - kv.float()).abs()
    s = scales.float()[:, None]
    sat = (kv.float().abs().amax(dim=1, keepdim=True) > 127.5 * 512)
    assert bool((err <= torch.where(sat, s, s / 2)).all())
    rng = np.random.Generator(np.random.PCG64(9701))
    rows = np.unique(np.r_[0:64, n - 64:n, rng.integers(0, n, 2000)])
    sample = kv[torch.from_numpy(rows).cuda()].cpu().numpy()
    rq, rs = oracle.kv_encode(sample)
    assert np.array_equal(codes[torch.from_numpy(rows).cuda()].cpu().numpy(), rq)
    assert np.array_equal(scales[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16), rs.view(np.uint16))


def test_kv_codec_argument_errors(q):
    import torch

    kv = torch.zeros((4, 128), dtype=torch.float16, device="cuda")
    c = torch.zeros((4, 128), dtype=torch.int8, device="cuda")
    s = torch.zeros(4, dtype=torch.float16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert q.lib.jllm_kv_encode_i8(kv.data_ptr(), c.data_ptr(), s.data_ptr(), 4, 96, st) == 2
    assert q.lib.jllm_kv_encode_i8(kv.data_ptr(), c.data_ptr(), s.data_ptr(), 0, 128, st) == 1
    assert q.lib.jllm_kv_encode_i8(None, c.data_ptr(), s.data_ptr(), 4, 128, st) == 1
    assert q.lib.jllm_kv_encode_i8(kv.data_ptr() + 2, c.data_ptr(), s.data_ptr(), 1, 128, st) == 3
    assert q.lib.jllm_kv_decode_i8(c.data_ptr(), s.data_ptr() + 1, kv.data_ptr(), 4, 128, st) == 3

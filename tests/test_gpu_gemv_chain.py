"""jllm_q4k_gemv_chain: a sequence of decode GEMV steps in one persistent launch.

Every output is compared with the fp64 oracle on the same seeded inputs, within
the matmul bound 2e-3 * sum|x*w| + 1e-5.  The step shapes cover what the kernel
splits differently: K from one block to the largest allowed (12288), odd block
counts, 1..4 matrices per step, matrices with fewer rows than there are SMs (so
that most CTAs own no row), empty matrices, and steps whose rows cut a CTA's
range at matrix boundaries.  The dependent chain feeds each step's fp16 output
to the next step as x, with every output filled with NaN before the call, so a
step that read its x before the previous step had written it shows as NaN or as
a mismatch with the oracle evaluated on the x the GPU actually produced."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import LAYER_SHAPES, assert_within, dev, oracle_matmul_rows, sample_cols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def scaled_q4k(w, k):
    """The Q4_K matrix w with d and dmin of every block multiplied by 2^-k (an input
    transform: the oracle reads the same bytes)."""
    b = np.array(w, copy=True).reshape(-1, 144)
    for off in (0, 2):
        v = b[:, off:off + 2].copy().view(np.float16).astype(np.float32) * np.float32(2.0 ** -k)
        b[:, off:off + 2] = v.astype(np.float16).view(np.uint8).reshape(-1, 2)
    return b.reshape(w.shape)


MIXED = [  # (K, [N per matrix])
    (256, [1, 7, 300, 0]),
    (2560, [4096, 1024, 1024]),
    (768, [33, 5000]),
    (12288, [100]),
    (2816, [0, 19]),
    (9728, [2560]),
    (4096, [151, 152, 153, 2]),
]


def test_mixed_steps(q):
    import torch

    steps, refs = [], []
    for i, (K, Ns) in enumerate(MIXED):
        x = synthetic.activations(1, K, synthetic.activation_seed(7, i, 0))
        ws = [synthetic.q4k_weights(n, K, synthetic.weight_seed(7, i, j)) if n else np.zeros((0, K // 256 * 144), np.uint8)
              for j, n in enumerate(Ns)]
        refs.append([oracle.matmul(w, x, n, K) if n else None for w, n in zip(ws, Ns)])
        ys = [torch.empty(max(n, 1), dtype=torch.float32, device="cuda")[:n] for n in Ns]
        steps.append(([dev(w) for w in ws], dev(x.reshape(K)), ys, Ns, K))
    chain = q.GemvChain(steps)
    for rnd in range(3):  # repeated: each call must leave the sync words zero for the next
        for _, _, ys, _, _ in steps:
            for y in ys:
                y.fill_(float("nan"))
        chain()
        assert q.jllm_get_device_error() == 0
        for i, ((K, Ns), (_, _, ys, _, _)) in enumerate(zip(MIXED, steps)):
            for j, n in enumerate(Ns):
                if n:
                    ref, s = refs[i][j]
                    assert_within(ys[j].cpu().numpy()[None, :], ref, s, f"round {rnd} step {i} matrix {j}")
    assert not chain.sync.any().item(), "sync words not returned to zero"


def test_dependent_chain_fp16(q):
    """x of step s+1 is the fp16 output of step s (2560 -> 4096 -> 9728 -> 2560 -> 512)."""
    import torch

    dims, shifts = [2560, 4096, 9728, 2560, 512], [5, 10, 11, 9]
    ws = [scaled_q4k(synthetic.q4k_weights(dims[i + 1], dims[i], synthetic.weight_seed(8, 0, i)), shifts[i])
          for i in range(4)]
    x0 = synthetic.activations(1, dims[0], synthetic.activation_seed(8, 0, 0))
    wd = [dev(w) for w in ws]
    outs = [torch.empty(dims[i + 1], dtype=torch.float16 if i < 3 else torch.float32, device="cuda") for i in range(4)]
    xs = [dev(x0.reshape(-1))] + outs[:3]
    chain = q.GemvChain([([wd[i]], xs[i], [outs[i]], [dims[i + 1]], dims[i]) for i in range(4)])
    for rnd in range(3):
        for o in outs:
            o.fill_(float("nan"))
        chain()
        assert q.jllm_get_device_error() == 0
        x_in = x0.reshape(1, -1)
        for i in range(4):
            y = outs[i].float().cpu().numpy()[None, :]
            ref, s = oracle.matmul(ws[i], x_in, dims[i + 1], dims[i])  # on the x the GPU produced
            assert_within(y, ref, s, f"round {rnd} step {i}")
            x_in = outs[i].cpu().numpy()[None, :] if i < 3 else None


def test_chain_in_cuda_graph(q):
    """The chain captured in a CUDA graph and replayed back to back."""
    import torch

    K, Ns = 2560, [4096, 1024, 1024]
    x = synthetic.activations(1, K, synthetic.activation_seed(9, 0, 0))
    ws = [synthetic.q4k_weights(n, K, synthetic.weight_seed(9, 0, j)) for j, n in enumerate(Ns)]
    ys = [torch.empty(n, dtype=torch.float32, device="cuda") for n in Ns]
    step = ([dev(w) for w in ws], dev(x.reshape(K)), ys, Ns, K)
    chain = q.GemvChain([step] * 8)  # eight dependent repeats of one step
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        chain(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain(s)
    for y in ys:
        y.fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert q.jllm_get_device_error() == 0
    for j, n in enumerate(Ns):
        ref, sref = oracle.matmul(ws[j], x, n, K)
        assert_within(ys[j].cpu().numpy()[None, :], ref, sref, f"graph matrix {j}")


def test_decode_sweep_full_size(q):
    """The 36-layer decode sweep as one chain (144 steps: q/k/v, o, gate/up, down),
    sampled rows of every matrix against the oracle."""
    import torch

    groups = (((0, 1, 2)), ((3,)), ((4, 5)), ((6,)))
    steps, samples = [], []
    rng = np.random.Generator(np.random.PCG64(11))
    for layer in range(synthetic.N_LAYERS):
        for gi, members in enumerate(groups):
            K = LAYER_SHAPES[members[0]][1]
            x = synthetic.activations(1, K, synthetic.activation_seed(1, layer * 8 + gi))
            ws, ys, Ns = [], [], []
            for m in members:
                name, _, N = LAYER_SHAPES[m]
                w = synthetic.q4k_weights(N, K, synthetic.weight_seed(1, layer, m))
                ws.append(dev(w))
                ys.append(torch.full((N,), float("nan"), dtype=torch.float32, device="cuda"))
                Ns.append(N)
                if layer in (0, 17, 35):  # three layers checked (first, middle, last)
                    samples.append((w, x, N, K, len(steps), len(Ns) - 1, sample_cols(N, rng)))
            steps.append((ws, dev(x.reshape(K)), ys, Ns, K))
    q.GemvChain(steps)()
    torch.cuda.synchronize()
    assert q.jllm_get_device_error() == 0
    for w, x, N, K, si, j, cols in samples:
        ref, s = oracle_matmul_rows(w, x, N, K, cols)
        y = steps[si][2][j].cpu().numpy()[cols][None, :]
        assert_within(y, ref, s, f"step {si} matrix {j}")
    for _, _, ys, _, _ in steps:  # every output written
        for y in ys:
            assert torch.isfinite(y).all().item()


@pytest.mark.parametrize("seed", [21, 22, 23])
def test_random_chains(q, seed):
    """Random small chains: 1..12 steps, K from one to eleven blocks, 1..4 matrices of
    0..700 rows, fp32 or fp16 outputs, every output against the oracle."""
    import torch

    rng = np.random.Generator(np.random.PCG64(seed))
    steps, refs = [], []
    for i in range(int(rng.integers(1, 13))):
        K = 256 * int(rng.integers(1, 12))
        cnt = int(rng.integers(1, 5))
        Ns = [int(rng.integers(0, 701)) for _ in range(cnt)]
        if sum(Ns) == 0:
            Ns[0] = 1
        f16 = bool(rng.integers(0, 2))
        x = synthetic.activations(1, K, synthetic.activation_seed(seed, i, 0))
        ws = [synthetic.q4k_weights(n, K, synthetic.weight_seed(seed, i, j)) if n
              else np.zeros((0, K // 256 * 144), np.uint8) for j, n in enumerate(Ns)]
        refs.append([oracle.matmul(w, x, n, K) if n else None for w, n in zip(ws, Ns)])
        dt = torch.float16 if f16 else torch.float32
        ys = [torch.full((max(n, 1),), float("nan"), dtype=dt, device="cuda")[:n] for n in Ns]
        steps.append(([dev(w) for w in ws], dev(x.reshape(K)), ys, Ns, K))
    q.GemvChain(steps)()
    assert q.jllm_get_device_error() == 0
    for i, (_, _, ys, Ns, K) in enumerate(steps):
        for j, n in enumerate(Ns):
            if n:
                ref, s_ = refs[i][j]
                y = ys[j].float().cpu().numpy()[None, :]
                assert_within(y, ref, s_, f"seed {seed} step {i} matrix {j} (K {K}, N {n})")

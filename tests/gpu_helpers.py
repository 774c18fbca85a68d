"""Shared helpers of the GPU parity tests (inputs from `synthetic`, expected
values from `oracle` only)."""
import numpy as np

import oracle
import synthetic

LAYER_SHAPES = synthetic.LAYER_SHAPES


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y, ref, s, label):
    """Every element of y within the matmul bound 2e-3*S + 1e-5 of the fp64 oracle."""
    y = np.asarray(y, dtype=np.float64)
    assert y.shape == ref.shape, (label, y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{label}: non-finite outputs"
    err = np.abs(y - ref)
    tol = oracle.tolerance(s)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{label}: {int(bad.sum())} of {bad.size} outside the bound; worst at {i}: "
                             f"got {y[i]!r} ref {ref[i]!r} err {err[i]:.3e} tol {tol[i]:.3e}")


def sample_cols(N, rng, n_random=64, edge=32, tile=128):
    cols = set(range(min(edge, N))) | set(range(max(0, N - edge), N))
    tail0 = (N // tile) * tile
    cols |= set(range(tail0, N))  # every column of a partial last tile
    cols |= set(rng.integers(0, N, size=min(n_random, N)).tolist())
    return np.array(sorted(cols), dtype=np.int64)


def sample_rows(M, rng, n_random=256, edge=128):
    if M <= 2 * edge + n_random:
        return np.arange(M)
    rows = set(range(edge)) | set(range(M - edge, M)) | set(rng.integers(0, M, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)

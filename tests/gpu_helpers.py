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


def oracle_matmul_rows(w, x, N, K, cols=None, threads=None):
    """oracle.matmul (or matmul_cols) over chunks of the rows of x on several host threads.
    The oracle itself stays single-threaded: each thread makes one ordinary oracle call on
    its own rows (ctypes releases the GIL), and the results are stacked in row order."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    x = np.asarray(x).reshape(-1, K)
    M = x.shape[0]
    threads = threads or min(16, os.cpu_count() or 1, M)
    bounds = np.linspace(0, M, threads + 1).astype(int)
    chunks = [(bounds[i], bounds[i + 1]) for i in range(threads) if bounds[i + 1] > bounds[i]]

    def one(c):
        xs = x[c[0]:c[1]]
        return oracle.matmul(w, xs, N, K) if cols is None else oracle.matmul_cols(w, xs, N, K, cols)

    with ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(one, chunks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def chained_bound(w, h_ref, t, N, K, cols=None):
    """Bound on |y - y_ref| for y = the GPU matmul of an input h_gpu with |h_gpu - h_ref| <= t
    elementwise, y_ref the exact matmul of h_ref: the matmul bound on h_gpu plus the
    propagated input error,
        2e-3 * sum_k |w_nk| (|h_ref,k| + t_k) + 1e-5 + sum_k |w_nk| t_k.
    Every term is an oracle quantity (the sums are the oracle's S of non-negative inputs)."""
    a = np.abs(np.asarray(h_ref, dtype=np.float64)) + t
    _, s_a = oracle_matmul_rows(w, a, N, K, cols)
    _, s_t = oracle_matmul_rows(w, np.asarray(t, dtype=np.float64), N, K, cols)
    return 2e-3 * s_a + 1e-5 + s_t

"""Edge-case inputs of the matmul parity tests: weight matrices whose rows mix
uniform random Q4_K blocks with closed-form blocks, and activations that mix
N(0,1) values with tiny ones and fp16 subnormals.

Test infrastructure only.  Blocks are assembled from fields with the oracle's
scale packer (pinned by tests/test_oracle_pins.py); nothing here comes from the
GPU path.  Row kinds (every block of the row):

  0 random (as in the synthetic workloads)
  1 all codes 0, every m_j = 0, every sc_j = 63, d = 2^-8   -> row of exact zeros
  2 all codes 15, every sc_j = 63, m_j random, d, dmin random
  3 d = dmin = 0, scales, mins and codes random             -> row of exact zeros
  4 any finite fp16 d and dmin (random sign, magnitude below a cap), rest random
  5 even sub-blocks zero (codes 0, m_j = 0), odd ones random
  6 all codes 0, m_j random (every weight -dmin*m_j)
  7 fp16-subnormal d and dmin, rest random
"""
from __future__ import annotations

import numpy as np

import oracle
import synthetic

N_KINDS = 8
# Largest magnitude bit pattern below 64.0 (0x5400): keeps |d*sc*q - dmin*m| <= 64*945
# within the fp16 range, the operand type of the tensor-core path.
CAP_FP16_OPERAND = 0x5400
CAP_FINITE = 0x7C00


def _set_header(blk, d_bits, dmin_bits):
    blk[0:2] = np.array([d_bits], dtype="<u2").view(np.uint8)
    blk[2:4] = np.array([dmin_bits], dtype="<u2").view(np.uint8)


def edge_weights(N: int, K: int, seed: int, cap_bits: int = CAP_FP16_OPERAND, kinds=None) -> np.ndarray:
    """[N, K/256*144] Q4_K bytes; row n has kind kinds[n] (default n % 8)."""
    nb = K // 256
    w = synthetic.q4k_weights(N, K, seed).reshape(N, nb, 144).copy()
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x5EED))
    if kinds is None:
        kinds = np.arange(N) % N_KINDS
    half = lambda v: int(np.array([v], dtype=np.float16).view(np.uint16)[0])
    for n in range(N):
        kind = int(kinds[n])
        for b in range(nb):
            blk = w[n, b]
            sc = rng.integers(0, 64, size=8)
            m = rng.integers(0, 64, size=8)
            if kind == 1:
                blk[16:] = 0
                blk[4:16] = oracle.pack_scale_min(np.full(8, 63), np.zeros(8, dtype=np.int64))
                _set_header(blk, half(2.0**-8), blk[2] | (blk[3] << 8))
            elif kind == 2:
                blk[16:] = 0xFF
                blk[4:16] = oracle.pack_scale_min(np.full(8, 63), m)
            elif kind == 3:
                _set_header(blk, 0, 0)
            elif kind == 4:
                bits = rng.integers(0, cap_bits, size=2) | (rng.integers(0, 2, size=2) << 15)
                _set_header(blk, int(bits[0]), int(bits[1]))
            elif kind == 5:
                m[0::2] = 0
                blk[4:16] = oracle.pack_scale_min(sc, m)
                for c in range(4):  # sub-block 2c = low nibbles of qs[32c .. 32c+31]
                    blk[16 + 32 * c:16 + 32 * c + 32] &= 0xF0
            elif kind == 6:
                blk[16:] = 0
                blk[4:16] = oracle.pack_scale_min(sc, m)
            elif kind == 7:
                bits = rng.integers(1, 0x400, size=2)
                _set_header(blk, int(bits[0]), int(bits[1]))
    return w.reshape(N, nb * 144)


def mixed_activations(M: int, K: int, seed: int) -> np.ndarray:
    """fp16 [M, K]: N(0,1), with a third of the entries ~1e-4 * N(0,1), a sixth random
    fp16 subnormals (either sign) and a few exact zeros."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(size=(M, K))
    u = rng.uniform(size=(M, K))
    x = np.where(u < 1 / 3, x * 1e-4, x).astype(np.float16)
    sub = (rng.integers(1, 0x400, size=(M, K)) | (rng.integers(0, 2, size=(M, K)) << 15)).astype(np.uint16)
    x = np.where((u >= 1 / 3) & (u < 0.5), sub.view(np.float16), x)
    x = np.where(u > 0.995, np.float16(0.0), x)
    return x.astype(np.float16)

"""Seeded synthetic inputs for the Q4_K matmul: the one module that both the
CPU oracle's tests and the GPU path's tests/benchmark draw inputs from.

It holds none of the method's arithmetic: it draws random bytes and random
fp16 activations, nothing else.  The Qwen3-4B Q4_K_M weights and prompts of
the genie-ai-runtime README ("Performance" and the CLI sample) are not
available, so these stand in for them:

* Weights: every super-block is 144 bytes in the GGUF Q4_K layout.  d and dmin
  are drawn uniformly (linear) in [2^-12, 2^-8] and rounded to the nearest
  fp16; the 12 packed scale/min bytes and the 128 code bytes are uniform
  random bytes.  Each of the 96 scale bits feeds exactly one bit of exactly
  one of the sixteen 6-bit fields (8 scales sc_j, 8 mins m_j), so uniform
  bytes are the same draw as independent uniform sc_j, m_j in 0..63.
* Activations: fp16 N(0, 1) from numpy's normal generator,
  optionally each token row scaled by U[0.5, 2] before rounding to fp16.

Random numbers come from numpy's PCG64 generator, seeded per tensor.
"""
from __future__ import annotations

import numpy as np

QK = 256
BLOCK_BYTES = 144

# Qwen3-4B layer shapes (K -> N): hidden 2560, 32 query heads and 8 KV heads
# of 128, MLP 9728 (genie-ai-runtime README CLI sample: 36 layers, 32 heads,
# 8 KV heads, 2560 dim).
LAYER_SHAPES = (
    ("q", 2560, 4096),
    ("k", 2560, 1024),
    ("v", 2560, 1024),
    ("o", 4096, 2560),
    ("gate", 2560, 9728),
    ("up", 2560, 9728),
    ("down", 9728, 2560),
)
N_LAYERS = 36
LM_HEAD = ("lm_head", 2560, 151936)


def weight_seed(config: int, layer: int, shape_index: int) -> int:
    """Seed of one weight tensor: config, layer and position in LAYER_SHAPES."""
    return 0x51344B00 + 4096 * config + 16 * layer + shape_index


def activation_seed(config: int, M: int, tag: int = 0) -> int:
    return 0x58000000 + 100000 * config + 16 * M + tag


def q4k_weights(N: int, K: int, seed: int) -> np.ndarray:
    """Random Q4_K weight tensor [N rows][K/256 blocks][144 bytes] as uint8 [N, K/256*144]."""
    if K % QK:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.integers(0, 256, size=(N, nb, BLOCK_BYTES), dtype=np.uint8)
    dd = rng.uniform(2.0**-12, 2.0**-8, size=(N, nb, 2)).astype("<f2")
    w[:, :, 0:4] = dd.view(np.uint8).reshape(N, nb, 4)  # little-endian d, dmin
    return w.reshape(N, nb * BLOCK_BYTES)


def activations(M: int, K: int, seed: int, per_token_scale: bool = False) -> np.ndarray:
    """fp16 [M, K] activations ~ N(0,1), rows optionally scaled by U[0.5, 2]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(size=(M, K))
    if per_token_scale:
        x *= rng.uniform(0.5, 2.0, size=(M, 1))
    return x.astype(np.float16)

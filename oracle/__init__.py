"""CPU oracle for the Q4_K dequant-fused matmul (ctypes wrapper over q4k_oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline / reference leg may import this module; the GPU
library (``bit_q4_weight_gb300``) never does, and the two share no source.

Every function restates a definition in plain single-threaded C, fp64:

* ``dequant``  -- the Q4_K super-block decode w = d*sc_j*q - dmin*m_j (public
  GGUF Q4_K layout; the genie-ai-runtime README, "At a glance", says the
  runtime loads GGUF Q4_K_M models but does not print the layout), rounded
  once to fp32, and from fp32 to fp16 for the fp16 output.
* ``matmul`` / ``matmul_cols`` -- y = X * dequant(W)^T in fp64 with k ascending,
  plus the error scale S = sum_k |x_k * w_nk| of the tolerance
  |y - y_ref| <= 2e-3 * S + 1e-5 (the "INT4 dequant-fused GEMV" and
  "tensor-core MMQ Q4_K prefill" of the README's Kernels bullet).
* ``swiglu`` -- h = silu(g) * u, silu(z) = z / (1 + e^-z) (the SwiGLU of the
  README's "fused RMSNorm + RoPE + SwiGLU" kernel).
* ``rmsnorm`` -- xn = x * gamma / sqrt(mean(x^2) + eps) per token row (the
  RMSNorm of the same kernel bullet; the standard root-mean-square norm, named
  but not printed on the pages), the prologue of the fused-norm GEMV.
* ``rope`` -- rotary position embedding of head vectors (pairs (i, i + D/2),
  angle pos * base^(-2i/D)), the RoPE of the same kernel bullet; the pages
  print no formula, this is the form of the Qwen3 model they run.
  ``head_rmsnorm`` -- ``rmsnorm`` applied per head vector (Qwen3's q/k norm).
* ``kv_encode`` / ``kv_decode`` -- the FP16 <-> INT8 KV codec of the README's KV
  cache bullet (per-vector power-of-two scale, round half to even; the rule and
  why it is drift-free are in q4k_oracle.c; the pages give no granularity).
* ``quantize`` -- a plain non-iterative quantiser used only for the round-trip
  pin (not on the pages; the rule is stated in q4k_oracle.c).

Pins: tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_q4k.so")
_lib = None

BLOCK_BYTES = 144
QK = 256


def build(force: bool = False) -> str:
    """Compile q4k_oracle.c into liboracle_q4k.so next to it (gcc, -O2, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oq_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oq_half_to_double.restype = ctypes.c_double
    lib.oq_float_to_half_rne.argtypes = [ctypes.c_float]
    lib.oq_float_to_half_rne.restype = ctypes.c_uint16
    lib.oq_scale_min.argtypes = [P, ctypes.c_int, P, P]
    lib.oq_scale_min.restype = None
    lib.oq_pack_scale_min.argtypes = [P, P, P]
    lib.oq_pack_scale_min.restype = None
    lib.oq_decode_block.argtypes = [P, P]
    lib.oq_decode_block.restype = None
    lib.oq_dequant.argtypes = [P, I64, I64, ctypes.c_int, P]
    lib.oq_dequant.restype = None
    lib.oq_matmul.argtypes = [P, P, I64, I64, I64, P, P]
    lib.oq_matmul.restype = ctypes.c_int
    lib.oq_matmul_cols.argtypes = [P, P, I64, I64, P, I64, P, P]
    lib.oq_matmul_cols.restype = ctypes.c_int
    lib.oq_swiglu.argtypes = [P, P, I64, P]
    lib.oq_swiglu.restype = None
    lib.oq_rmsnorm.argtypes = [P, P, I64, I64, ctypes.c_double, P]
    lib.oq_rmsnorm.restype = None
    lib.oq_rope.argtypes = [P, I64, I64, I64, ctypes.c_double, P]
    lib.oq_rope.restype = None
    lib.oq_kv_encode.argtypes = [P, I64, I64, P, P]
    lib.oq_kv_encode.restype = None
    lib.oq_kv_decode.argtypes = [P, P, I64, I64, P]
    lib.oq_kv_decode.restype = None
    lib.oq_quantize_block.argtypes = [P, P]
    lib.oq_quantize_block.restype = None
    lib.oq_quantize.argtypes = [P, I64, I64, P]
    lib.oq_quantize.restype = None
    lib.oq_half_to_double_n.argtypes = [P, I64, P]
    lib.oq_half_to_double_n.restype = None
    lib.oq_float_to_half_rne_n.argtypes = [P, I64, P]
    lib.oq_float_to_half_rne_n.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_w(w: np.ndarray, N: int, K: int) -> np.ndarray:
    if K % QK:
        raise ValueError("K must be a multiple of 256")
    w = np.ascontiguousarray(w, dtype=np.uint8)
    if w.size != N * (K // QK) * BLOCK_BYTES:
        raise ValueError("W must hold N*K/256 blocks of 144 bytes")
    return w


def half_bits_to_double(h: np.ndarray) -> np.ndarray:
    """binary16 bit patterns (uint16) -> exact fp64 values."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oq_half_to_double_n(_ptr(h), h.size, _ptr(out))
    return out


def float_to_half_bits(f: np.ndarray) -> np.ndarray:
    """fp32 -> binary16 bit patterns, round to nearest even (the oracle's own routine)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().oq_float_to_half_rne_n(_ptr(f), f.size, _ptr(out))
    return out


def scale_min(s12: bytes | np.ndarray, j: int) -> tuple[int, int]:
    """(sc_j, m_j) of sub-block j from the 12 packed scale bytes."""
    s = np.ascontiguousarray(np.frombuffer(bytes(s12), dtype=np.uint8) if isinstance(s12, (bytes, bytearray)) else s12, dtype=np.uint8)
    sc = ctypes.c_int()
    m = ctypes.c_int()
    _load().oq_scale_min(_ptr(s), int(j), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def pack_scale_min(sc, m) -> np.ndarray:
    """Pack eight (sc_j, m_j) pairs (0..63) into 12 bytes."""
    sc = np.ascontiguousarray(sc, dtype=np.int32)
    m = np.ascontiguousarray(m, dtype=np.int32)
    out = np.zeros(12, dtype=np.uint8)
    _load().oq_pack_scale_min(_ptr(sc), _ptr(m), _ptr(out))
    return out


def decode_block(blk) -> np.ndarray:
    """One 144-byte super-block -> its 256 exact values (fp64)."""
    b = np.ascontiguousarray(np.frombuffer(bytes(blk), dtype=np.uint8) if isinstance(blk, (bytes, bytearray)) else blk, dtype=np.uint8)
    if b.size != BLOCK_BYTES:
        raise ValueError("a block is 144 bytes")
    out = np.empty(QK, dtype=np.float64)
    _load().oq_decode_block(_ptr(b), _ptr(out))
    return out


def dequant(w: np.ndarray, N: int, K: int, out_dtype: str = "f32") -> np.ndarray:
    """dequant(W) as an [N, K] array: fp32 values, or fp16 (returned as np.float16)."""
    w = _check_w(w, N, K)
    if out_dtype == "f32":
        out = np.empty((N, K), dtype=np.float32)
        _load().oq_dequant(_ptr(w), N, K, 0, _ptr(out))
        return out
    if out_dtype == "f16":
        out = np.empty((N, K), dtype=np.uint16)
        _load().oq_dequant(_ptr(w), N, K, 1, _ptr(out))
        return out.view(np.float16)
    raise ValueError("out_dtype must be 'f32' or 'f16'")


def matmul(w: np.ndarray, x: np.ndarray, N: int, K: int) -> tuple[np.ndarray, np.ndarray]:
    """fp64 y[M,N] = x[M,K] * dequant(W)^T and S[M,N] = sum_k |x*w| (x any float dtype, converted exactly)."""
    w = _check_w(w, N, K)
    x = np.ascontiguousarray(np.asarray(x).reshape(-1, K), dtype=np.float64)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    s = np.empty((M, N), dtype=np.float64)
    if _load().oq_matmul(_ptr(w), _ptr(x), M, N, K, _ptr(y), _ptr(s)) != 0:
        raise MemoryError("oracle matmul: out of memory")
    return y, s


def matmul_cols(w: np.ndarray, x: np.ndarray, N: int, K: int, cols) -> tuple[np.ndarray, np.ndarray]:
    """Like matmul but only for output columns ``cols``; returns [M, len(cols)] arrays."""
    w = _check_w(w, N, K)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if cols.size and (cols.min() < 0 or cols.max() >= N):
        raise IndexError("column out of range")
    x = np.ascontiguousarray(np.asarray(x).reshape(-1, K), dtype=np.float64)
    M = x.shape[0]
    y = np.empty((M, cols.size), dtype=np.float64)
    s = np.empty((M, cols.size), dtype=np.float64)
    if _load().oq_matmul_cols(_ptr(w), _ptr(x), M, K, _ptr(cols), cols.size, _ptr(y), _ptr(s)) != 0:
        raise MemoryError("oracle matmul: out of memory")
    return y, s


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u in fp64."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    if g.shape != u.shape:
        raise ValueError("g and u must have the same shape")
    h = np.empty(g.shape, dtype=np.float64)
    _load().oq_swiglu(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """xn = x * gamma / sqrt(mean(x^2) + eps) per row, fp64 ([M, K] or [K])."""
    gamma = np.ascontiguousarray(gamma, dtype=np.float64).reshape(-1)
    K = gamma.size
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1, K))
    out = np.empty_like(xa)
    _load().oq_rmsnorm(_ptr(xa), _ptr(gamma), xa.shape[0], K, float(eps), _ptr(out))
    return out.reshape(np.asarray(x).shape)


def rope(v: np.ndarray, pos: int, base: float, head_dim: int = 128) -> np.ndarray:
    """Rotary position embedding of head vectors ([..., head_dim] fp64; pairs (i, i + head_dim/2),
    angle pos * base^(-2i/head_dim)), fp64."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    va = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    if va.size % head_dim:
        raise ValueError("size must be a multiple of head_dim")
    out = np.empty_like(va)
    _load().oq_rope(_ptr(va), va.size // head_dim, head_dim, int(pos), float(base), _ptr(out))
    return out


def head_rmsnorm(v: np.ndarray, gamma: np.ndarray, eps: float, head_dim: int = 128) -> np.ndarray:
    """RMSNorm of every head vector of v (the per-head q/k norm that Qwen3 applies before
    RoPE): ``rmsnorm`` on v viewed as [heads, head_dim] rows, gamma [head_dim]."""
    va = np.asarray(v, dtype=np.float64)
    return rmsnorm(va.reshape(-1, head_dim), gamma, eps).reshape(va.shape)


def kv_encode(v: np.ndarray, dim: int = 128) -> tuple[np.ndarray, np.ndarray]:
    """INT8 KV codec: fp16 vectors of `dim` values -> (int8 codes [..., dim], fp16 power-of-two
    scales [...]); see oq_kv_encode for the rule."""
    va = np.ascontiguousarray(np.asarray(v, dtype=np.float16))
    if va.size % dim:
        raise ValueError("size must be a multiple of dim")
    n = va.size // dim
    q = np.empty(va.shape, dtype=np.int8)
    sc = np.empty(n, dtype=np.uint16)
    _load().oq_kv_encode(_ptr(va.view(np.uint16)), n, dim, _ptr(q), _ptr(sc))
    return q, sc.view(np.float16).reshape(va.shape[:-1] if va.ndim > 1 and va.shape[-1] == dim else (n,))


def kv_decode(q: np.ndarray, scales: np.ndarray, dim: int = 128) -> np.ndarray:
    """INT8 KV codec: codes and scales -> fp16 values q * scale."""
    qa = np.ascontiguousarray(np.asarray(q, dtype=np.int8))
    sa = np.ascontiguousarray(np.asarray(scales, dtype=np.float16)).view(np.uint16)
    n = qa.size // dim
    if qa.size % dim or sa.size != n:
        raise ValueError("one scale per vector of dim codes")
    out = np.empty(qa.shape, dtype=np.uint16)
    _load().oq_kv_decode(_ptr(qa), _ptr(sa), n, dim, _ptr(out))
    return out.view(np.float16)


def quantize(w: np.ndarray) -> np.ndarray:
    """Quantise an [N, K] fp64 matrix into Q4_K blocks ([N, K/256*144] bytes)."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    N, K = w.shape
    if K % QK:
        raise ValueError("K must be a multiple of 256")
    out = np.empty((N, K // QK * BLOCK_BYTES), dtype=np.uint8)
    _load().oq_quantize(_ptr(w), N, K, _ptr(out))
    return out


def tolerance(s: np.ndarray) -> np.ndarray:
    """The matmul's per-element bound: 2e-3 * S + 1e-5."""
    return 2e-3 * np.asarray(s, dtype=np.float64) + 1e-5


def swiglu_tolerance(g: np.ndarray, u: np.ndarray, sg: np.ndarray, su: np.ndarray) -> np.ndarray:
    """Per-element bound for a GPU h = fp16(silu(g') * u') whose g', u' each meet the matmul bound.

    With Eg = tolerance(sg), Eu = tolerance(su) and |silu'| <= 1.1 everywhere, the exact
    product of the perturbed inputs differs from silu(g)*u by at most
        P = 1.1*Eg*(|u| + Eu) + |silu(g)|*Eu,
    and the fp32 evaluation plus the rounding to fp16 add at most 2^-10 of its magnitude,
    |silu(g)*u| + P, so
        |h' - silu(g)*u| <= (1 + 2^-10)*P + 2^-10*|silu(g)*u| + 1e-5.
    """
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    eg = tolerance(sg)
    eu = tolerance(su)
    sil = g / (1.0 + np.exp(-np.clip(g, -700, 700)))
    pert = 1.1 * eg * (np.abs(u) + eu) + np.abs(sil) * eu
    return (1.0 + 2.0**-10) * pert + 2.0**-10 * np.abs(sil * u) + 1e-5

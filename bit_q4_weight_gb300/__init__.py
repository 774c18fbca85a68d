"""Python binding of libjllm_q4k.so, the GB300 (sm_103a) Q4_K dequant-fused matmul library.

Argument marshalling only: every function checks tensor dtypes, shapes,
devices and contiguity, allocates the output tensor when none is given, and
calls the C entry point of the same name (include/jllm_q4k.h) on the current
torch CUDA stream.  All computation happens in the library's CUDA kernels;
there is no CPU fallback, and importing this module fails loudly when the
library has not been built.

Layouts (see the header): W is uint8 [N, K/256*144] (GGUF Q4_K super-blocks,
rows contiguous), X is fp16 [M, K], Y is [M, N] fp32 or fp16.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

LIB_PATH = _build.LIB
BLOCK_BYTES = 144
QK = 256

# status codes (jllm_status)
JLLM_OK = 0
JLLM_ERR_INVALID_ARG = 1
JLLM_ERR_UNSUPPORTED_SHAPE = 2
JLLM_ERR_MISALIGNED = 3
JLLM_ERR_UNSUPPORTED_DTYPE = 4
JLLM_ERR_WORKSPACE = 5
JLLM_ERR_CUDA = 6
JLLM_ERR_DEVICE_TIMEOUT = 7
JLLM_ERR_NO_DEVICE = 8
# dtypes (jllm_dtype)
JLLM_F32 = 0
JLLM_F16 = 1

# Every symbol include/jllm_q4k.h declares.
EXPORTS = (
    "jllm_q4k_dequant",
    "jllm_q4k_gemv",
    "jllm_q4k_gemv_batch",
    "jllm_q4k_gemv_rmsnorm_batch",
    "jllm_q4k_gemv_qkv_rope",
    "jllm_q4k_gemv_chain",
    "jllm_q4k_gemv_chain_sync_bytes",
    "jllm_q4k_gemm",
    "jllm_q4k_gemm_noalloc",
    "jllm_q4k_gemm_batch",
    "jllm_q4k_ffn_swiglu",
    "jllm_kv_encode_i8",
    "jllm_kv_decode_i8",
    "jllm_q4k_workspace_bytes",
    "jllm_q4k_gemv_max_m",
    "jllm_get_device_error",
    "jllm_status_string",
)


class JllmError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
        "or python bit_q4_weight_gb300/_build.py)"
    )

lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_ST = ctypes.c_int

lib.jllm_q4k_dequant.argtypes = [_P, _P, ctypes.c_int, _I64, _I64, _P]
lib.jllm_q4k_dequant.restype = _ST
lib.jllm_q4k_gemv.argtypes = [_P, _P, _P, _I64, _I64, _P, _SZ, _P]
lib.jllm_q4k_gemv.restype = _ST
lib.jllm_q4k_gemv_batch.argtypes = [_P, _P, _P, ctypes.c_int, _P, _I64, _P]
lib.jllm_q4k_gemv_batch.restype = _ST
lib.jllm_q4k_gemv_rmsnorm_batch.argtypes = [_P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_float, _I64, _P]
lib.jllm_q4k_gemv_rmsnorm_batch.restype = _ST
lib.jllm_q4k_gemv_qkv_rope.argtypes = [_P, _P, _I64, _I64, _P, _I64, _P, ctypes.c_float, _P, _P, ctypes.c_float,
                                       _I64, ctypes.c_float, _P]
lib.jllm_q4k_gemv_qkv_rope.restype = _ST
CHAIN_MAX_STEPS = 256
CHAIN_MAX_MATS = 4
CHAIN_MAX_K = 12288


class GemvStep(ctypes.Structure):
    """jllm_gemv_step of the header."""
    _fields_ = [("count", ctypes.c_int32), ("y_f16", ctypes.c_int32), ("K", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("w_q4k", ctypes.c_void_p * CHAIN_MAX_MATS),
                ("y", ctypes.c_void_p * CHAIN_MAX_MATS), ("N", ctypes.c_int64 * CHAIN_MAX_MATS)]


lib.jllm_q4k_gemv_chain.argtypes = [ctypes.POINTER(GemvStep), ctypes.c_int, _P, _P]
lib.jllm_q4k_gemv_chain.restype = _ST
lib.jllm_q4k_gemv_chain_sync_bytes.argtypes = [ctypes.c_int]
lib.jllm_q4k_gemv_chain_sync_bytes.restype = _SZ
lib.jllm_q4k_gemm.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _P, _SZ, _P]
lib.jllm_q4k_gemm.restype = _ST
lib.jllm_q4k_gemm_noalloc.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _P]
lib.jllm_q4k_gemm_noalloc.restype = _ST
lib.jllm_q4k_gemm_batch.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _P, _I64, ctypes.c_int, _P, _SZ, _P]
lib.jllm_q4k_gemm_batch.restype = _ST
lib.jllm_q4k_ffn_swiglu.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]
lib.jllm_q4k_ffn_swiglu.restype = _ST
lib.jllm_kv_encode_i8.argtypes = [_P, _P, _P, _I64, _I64, _P]
lib.jllm_kv_encode_i8.restype = _ST
lib.jllm_kv_decode_i8.argtypes = [_P, _P, _P, _I64, _I64, _P]
lib.jllm_kv_decode_i8.restype = _ST
lib.jllm_q4k_workspace_bytes.argtypes = [_I64, _I64, _I64]
lib.jllm_q4k_workspace_bytes.restype = _SZ
lib.jllm_q4k_gemv_max_m.argtypes = []
lib.jllm_q4k_gemv_max_m.restype = ctypes.c_int
lib.jllm_get_device_error.argtypes = [_P]
lib.jllm_get_device_error.restype = _ST
lib.jllm_status_string.argtypes = [_ST]
lib.jllm_status_string.restype = ctypes.c_char_p


def status_string(status: int) -> str:
    return lib.jllm_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != JLLM_OK:
        raise JllmError(status, where)


# ------------------------------------------------------------ tensor helpers --

def _torch():
    import torch

    return torch


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _need(t, dtype, shape, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _w_shape(N: int, K: int):
    return (N, K // QK * BLOCK_BYTES)


# Zero-filled workspaces kept per (device, stream): the library returns a
# workspace to its reusable state after every call, and calls on one stream
# are ordered, so one buffer per stream suffices.
_WS_CACHE = {}


def _ws(M, N, K, ws, device, stream):
    need = int(lib.jllm_q4k_workspace_bytes(M, N, K))
    if need == 0 or ws is False:  # ws=False: run without a workspace
        return None, 0
    torch = _torch()
    if ws is None:
        key = (device.index if device.index is not None else torch.cuda.current_device(), _stream_ptr(stream))
        ws = _WS_CACHE.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(need, dtype=torch.uint8, device=device)
            _WS_CACHE[key] = ws
    return ws, ws.numel() * ws.element_size()


def workspace(M: int, N: int, K: int, device=None):
    """A zero-filled workspace tensor for gemm/ffn_swiglu of this shape (None if none is used)."""
    torch = _torch()
    need = int(lib.jllm_q4k_workspace_bytes(M, N, K))
    if need == 0:
        return None
    return torch.zeros(need, dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------ the API --

def jllm_q4k_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib.jllm_q4k_workspace_bytes(M, N, K))


def jllm_q4k_gemv_max_m() -> int:
    return int(lib.jllm_q4k_gemv_max_m())


def jllm_get_device_error(stream=None) -> int:
    """Synchronise the stream and return the device error status (0 = JLLM_OK)."""
    return int(lib.jllm_get_device_error(_stream_ptr(stream)))


def jllm_q4k_dequant(w, N: int, K: int, out_dtype=None, out=None, stream=None):
    """dequant(W) as an [N, K] fp32 (default) or fp16 tensor."""
    torch = _torch()
    out_dtype = out_dtype or (out.dtype if out is not None else torch.float32)
    if out_dtype not in (torch.float32, torch.float16):
        raise TypeError("out_dtype must be torch.float32 or torch.float16")
    _need(w, torch.uint8, _w_shape(N, K), "w")
    if out is None:
        out = torch.empty((N, K), dtype=out_dtype, device=w.device)
    _need(out, out_dtype, (N, K), "out")
    dt = JLLM_F16 if out_dtype == torch.float16 else JLLM_F32
    _check(lib.jllm_q4k_dequant(w.data_ptr(), out.data_ptr(), dt, N, K, _stream_ptr(stream)), "jllm_q4k_dequant")
    return out


def jllm_q4k_gemv(w, x, N: int, K: int, out=None, ws=None, stream=None):
    """y[N] (fp32) = dequant(W) x for one fp16 activation row x[K]."""
    torch = _torch()
    _need(w, torch.uint8, _w_shape(N, K), "w")
    if x.dim() == 2 and x.shape[0] == 1:
        x = x.view(K)
    _need(x, torch.float16, (K,), "x")
    if out is None:
        out = torch.empty((N,), dtype=torch.float32, device=w.device)
    _need(out, torch.float32, (N,), "out")
    ws, nbytes = _ws(1, N, K, ws, w.device, stream)
    _check(
        lib.jllm_q4k_gemv(w.data_ptr(), x.data_ptr(), out.data_ptr(), N, K,
                          ws.data_ptr() if ws is not None else None, nbytes, _stream_ptr(stream)),
        "jllm_q4k_gemv",
    )
    return out


def jllm_q4k_gemv_batch(ws_q4k, x, Ns, K: int, outs=None, stream=None):
    """[y_i[N_i] (fp32) = dequant(W_i) x] for up to 8 matrices sharing one fp16 x[K], one launch."""
    torch = _torch()
    ws_q4k, Ns = list(ws_q4k), [int(n) for n in Ns]
    if not 1 <= len(ws_q4k) <= 8 or len(Ns) != len(ws_q4k):
        raise ValueError("1 to 8 matrices, one row count each")
    for i, (w, n) in enumerate(zip(ws_q4k, Ns)):
        _need(w, torch.uint8, _w_shape(n, K), f"w[{i}]")
    if x.dim() == 2 and x.shape[0] == 1:
        x = x.view(K)
    _need(x, torch.float16, (K,), "x")
    if outs is None:
        outs = [torch.empty((n,), dtype=torch.float32, device=x.device) for n in Ns]
    for i, (o, n) in enumerate(zip(outs, Ns)):
        _need(o, torch.float32, (n,), f"out[{i}]")
    cnt = len(Ns)
    wp = (ctypes.c_void_p * cnt)(*[w.data_ptr() for w in ws_q4k])
    yp = (ctypes.c_void_p * cnt)(*[o.data_ptr() for o in outs])
    npa = (ctypes.c_int64 * cnt)(*Ns)
    _check(lib.jllm_q4k_gemv_batch(wp, yp, npa, cnt, x.data_ptr(), K, _stream_ptr(stream)), "jllm_q4k_gemv_batch")
    return outs


def jllm_q4k_gemv_rmsnorm_batch(ws_q4k, x, gamma, eps: float, Ns, K: int, outs=None, stream=None):
    """[y_i[N_i] (fp32) = dequant(W_i) rmsnorm(x)] for up to 8 matrices sharing one fp16 x[K];
    gamma fp32 [K]; the norm runs in the GEMV's prologue (one launch)."""
    torch = _torch()
    ws_q4k, Ns = list(ws_q4k), [int(n) for n in Ns]
    if not 1 <= len(ws_q4k) <= 8 or len(Ns) != len(ws_q4k):
        raise ValueError("1 to 8 matrices, one row count each")
    for i, (w, n) in enumerate(zip(ws_q4k, Ns)):
        _need(w, torch.uint8, _w_shape(n, K), f"w[{i}]")
    if x.dim() == 2 and x.shape[0] == 1:
        x = x.view(K)
    _need(x, torch.float16, (K,), "x")
    _need(gamma, torch.float32, (K,), "gamma")
    if outs is None:
        outs = [torch.empty((n,), dtype=torch.float32, device=x.device) for n in Ns]
    for i, (o, n) in enumerate(zip(outs, Ns)):
        _need(o, torch.float32, (n,), f"out[{i}]")
    cnt = len(Ns)
    wp = (ctypes.c_void_p * cnt)(*[w.data_ptr() for w in ws_q4k])
    yp = (ctypes.c_void_p * cnt)(*[o.data_ptr() for o in outs])
    npa = (ctypes.c_int64 * cnt)(*Ns)
    _check(lib.jllm_q4k_gemv_rmsnorm_batch(wp, yp, npa, cnt, x.data_ptr(), gamma.data_ptr(), float(eps), K,
                                           _stream_ptr(stream)), "jllm_q4k_gemv_rmsnorm_batch")
    return outs


def jllm_q4k_gemv_qkv_rope(w_qkv, x, n_q_heads: int, n_kv_heads: int, K: int, pos: int, rope_base: float = 1e6,
                           gamma=None, eps: float = 1e-6, q_gamma=None, k_gamma=None, head_eps: float = 1e-6,
                           outs=None, stream=None):
    """(q, k, v) fp32 of one fp16 token x[K]: the three projections in one launch, RoPE at `pos`
    on q and k (heads of 128), optional RMSNorm of x (gamma [K]) and per-head RMSNorm of q / k
    (q_gamma, k_gamma [128])."""
    torch = _torch()
    w_qkv = list(w_qkv)
    if len(w_qkv) != 3:
        raise ValueError("three matrices: Wq, Wk, Wv")
    Ns = [n_q_heads * 128, n_kv_heads * 128, n_kv_heads * 128]
    for i, (w, n) in enumerate(zip(w_qkv, Ns)):
        _need(w, torch.uint8, _w_shape(n, K), f"w[{i}]")
    if x.dim() == 2 and x.shape[0] == 1:
        x = x.view(K)
    _need(x, torch.float16, (K,), "x")
    for name, g, n in (("gamma", gamma, K), ("q_gamma", q_gamma, 128), ("k_gamma", k_gamma, 128)):
        if g is not None:
            _need(g, torch.float32, (n,), name)
    if outs is None:
        outs = [torch.empty((n,), dtype=torch.float32, device=x.device) for n in Ns]
    for i, (o, n) in enumerate(zip(outs, Ns)):
        _need(o, torch.float32, (n,), f"out[{i}]")
    wp = (ctypes.c_void_p * 3)(*[w.data_ptr() for w in w_qkv])
    yp = (ctypes.c_void_p * 3)(*[o.data_ptr() for o in outs])
    ptr = lambda t: t.data_ptr() if t is not None else None
    _check(lib.jllm_q4k_gemv_qkv_rope(wp, yp, n_q_heads, n_kv_heads, x.data_ptr(), K, ptr(gamma), float(eps),
                                      ptr(q_gamma), ptr(k_gamma), float(head_eps), int(pos), float(rope_base),
                                      _stream_ptr(stream)), "jllm_q4k_gemv_qkv_rope")
    return outs


def jllm_q4k_gemv_chain_sync_bytes(n_steps: int) -> int:
    return int(lib.jllm_q4k_gemv_chain_sync_bytes(int(n_steps)))


class GemvChain:
    """A jllm_q4k_gemv_chain call prepared once: `steps` is a sequence of
    (ws_q4k, x, outs, Ns, K) -- the matrices of a step (1..4 uint8 [N_i, K/256*144]
    tensors), its fp16 [K] x, its outputs (fp32 or fp16 [N_i], all one dtype) and
    row counts.  The descriptors are packed here, with a zeroed sync buffer owned
    by the object; calling it enqueues the whole chain (one launch).  The tensors
    must stay alive while the object is used."""

    def __init__(self, steps, device=None, sync=True):
        torch = _torch()
        steps = list(steps)
        n = len(steps)
        if not 1 <= n <= CHAIN_MAX_STEPS:
            raise ValueError(f"a chain has 1..{CHAIN_MAX_STEPS} steps, got {n}")
        self._arr = (GemvStep * n)()
        self._keep = []
        dev = None
        for i, (ws_q4k, x, outs, Ns, K) in enumerate(steps):
            cnt = len(ws_q4k)
            if not 1 <= cnt <= CHAIN_MAX_MATS or len(outs) != cnt or len(Ns) != cnt:
                raise ValueError(f"step {i}: 1..{CHAIN_MAX_MATS} matrices, as many outputs and row counts")
            _need(x, torch.float16, (K,), f"steps[{i}].x")
            f16 = outs[0].dtype == torch.float16
            st = self._arr[i]
            st.count, st.y_f16, st.K, st.x = cnt, int(f16), int(K), x.data_ptr()
            for j in range(cnt):
                _need(ws_q4k[j], torch.uint8, _w_shape(Ns[j], K), f"steps[{i}].w[{j}]")
                _need(outs[j], torch.float16 if f16 else torch.float32, (Ns[j],), f"steps[{i}].y[{j}]")
                st.w_q4k[j], st.y[j], st.N[j] = ws_q4k[j].data_ptr(), outs[j].data_ptr(), int(Ns[j])
            dev = x.device
        self.n_steps = n
        self.sync = _chain_sync(n, device or dev, False) if sync else None

    def __call__(self, stream=None):
        _check(lib.jllm_q4k_gemv_chain(self._arr, self.n_steps, self.sync.data_ptr(), _stream_ptr(stream)),
               "jllm_q4k_gemv_chain")


# Zeroed sync buffers of one-shot chains, per (device, stream, steps): a chain
# that completes leaves its buffer zeroed, and calls on one stream are ordered.
_SYNC_CACHE = {}


def _chain_sync(n, device, stream):
    """A zeroed sync buffer for n steps: private (stream None) or shared per stream."""
    torch = _torch()
    device = torch.device(device)
    idx = device.index if device.index is not None else torch.cuda.current_device()
    key = (idx, _stream_ptr(stream), n) if stream is not False else None
    buf = _SYNC_CACHE.get(key) if key else None
    if buf is None:
        buf = torch.zeros(jllm_q4k_gemv_chain_sync_bytes(n), dtype=torch.uint8, device=device)
        torch.cuda.synchronize(device)  # zero before any stream uses it
        if key:
            _SYNC_CACHE[key] = buf
    return buf


def jllm_q4k_gemv_chain(steps, stream=None):
    """One-shot jllm_q4k_gemv_chain over steps of (ws_q4k, x, outs, Ns, K) (see GemvChain);
    outs given as None are allocated (fp32).  Returns the outputs, one list per step."""
    torch = _torch()
    filled = []
    for ws_q4k, x, outs, Ns, K in steps:
        if outs is None:
            outs = [torch.empty(int(n), dtype=torch.float32, device=x.device) for n in Ns]
        filled.append((ws_q4k, x, outs, Ns, K))
    ch = GemvChain(filled, sync=False)
    ch.sync = _chain_sync(ch.n_steps, filled[0][1].device, stream)
    ch(stream)
    return [o for (_, _, o, _, _) in filled]


def jllm_q4k_gemm(w, x, N: int, K: int, out_dtype=None, out=None, ws=None, stream=None):
    """Y[M, N] = X[M, K] dequant(W)^T; fp32 (default) or fp16 output."""
    torch = _torch()
    _need(w, torch.uint8, _w_shape(N, K), "w")
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M = int(x.shape[0])
    _need(x, torch.float16, (M, K), "x")
    out_dtype = out_dtype or (out.dtype if out is not None else torch.float32)
    if out_dtype not in (torch.float32, torch.float16):
        raise TypeError("out_dtype must be torch.float32 or torch.float16")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=w.device)
    _need(out, out_dtype, (M, N), "out")
    ws, nbytes = _ws(M, N, K, ws, w.device, stream)
    dt = JLLM_F16 if out_dtype == torch.float16 else JLLM_F32
    _check(
        lib.jllm_q4k_gemm(w.data_ptr(), x.data_ptr(), out.data_ptr(), dt, M, N, K,
                          ws.data_ptr() if ws is not None else None, nbytes, _stream_ptr(stream)),
        "jllm_q4k_gemm",
    )
    return out


def jllm_q4k_gemm_noalloc(w, x, N: int, K: int, out_dtype=None, out=None, stream=None):
    """As jllm_q4k_gemm, with the library's static device workspace (no allocation)."""
    torch = _torch()
    _need(w, torch.uint8, _w_shape(N, K), "w")
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M = int(x.shape[0])
    _need(x, torch.float16, (M, K), "x")
    out_dtype = out_dtype or (out.dtype if out is not None else torch.float32)
    if out_dtype not in (torch.float32, torch.float16):
        raise TypeError("out_dtype must be torch.float32 or torch.float16")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=w.device)
    _need(out, out_dtype, (M, N), "out")
    dt = JLLM_F16 if out_dtype == torch.float16 else JLLM_F32
    _check(lib.jllm_q4k_gemm_noalloc(w.data_ptr(), x.data_ptr(), out.data_ptr(), dt, M, N, K, _stream_ptr(stream)),
           "jllm_q4k_gemm_noalloc")
    return out


def jllm_q4k_gemm_batch(ws_q4k, x, Ns, K: int, out_dtype=None, outs=None, ws=None, stream=None):
    """[Y_i[M, N_i] = X[M, K] dequant(W_i)^T] for up to 4 matrices sharing one fp16 X, one launch;
    fp32 (default) or fp16 outputs."""
    torch = _torch()
    ws_q4k, Ns = list(ws_q4k), [int(n) for n in Ns]
    if not 1 <= len(ws_q4k) <= 4 or len(Ns) != len(ws_q4k):
        raise ValueError("1 to 4 matrices, one row count each")
    for i, (w, n) in enumerate(zip(ws_q4k, Ns)):
        _need(w, torch.uint8, _w_shape(n, K), f"w[{i}]")
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M = int(x.shape[0])
    _need(x, torch.float16, (M, K), "x")
    out_dtype = out_dtype or (outs[0].dtype if outs else torch.float32)
    if out_dtype not in (torch.float32, torch.float16):
        raise TypeError("out_dtype must be torch.float32 or torch.float16")
    if outs is None:
        outs = [torch.empty((M, n), dtype=out_dtype, device=x.device) for n in Ns]
    for i, (o, n) in enumerate(zip(outs, Ns)):
        _need(o, out_dtype, (M, n), f"out[{i}]")
    ws, nbytes = _ws(M, sum(Ns), K, ws, x.device, stream)
    cnt = len(Ns)
    wp = (ctypes.c_void_p * cnt)(*[w.data_ptr() for w in ws_q4k])
    yp = (ctypes.c_void_p * cnt)(*[o.data_ptr() for o in outs])
    npa = (ctypes.c_int64 * cnt)(*Ns)
    dt = JLLM_F16 if out_dtype == torch.float16 else JLLM_F32
    _check(
        lib.jllm_q4k_gemm_batch(wp, x.data_ptr(), yp, dt, M, npa, K, cnt,
                                ws.data_ptr() if ws is not None else None, nbytes, _stream_ptr(stream)),
        "jllm_q4k_gemm_batch",
    )
    return outs


def jllm_kv_encode_i8(kv, head_dim: int = 128, codes=None, scales=None, stream=None):
    """fp16 KV vectors [..., head_dim] -> (int8 codes of the same shape, fp16 scales [...])."""
    torch = _torch()
    if kv.shape[-1] != head_dim:
        raise ValueError("last dimension must be head_dim")
    _need(kv, torch.float16, None, "kv")
    n = kv.numel() // head_dim
    if codes is None:
        codes = torch.empty(kv.shape, dtype=torch.int8, device=kv.device)
    if scales is None:
        scales = torch.empty(kv.shape[:-1], dtype=torch.float16, device=kv.device)
    _need(codes, torch.int8, kv.shape, "codes")
    _need(scales, torch.float16, kv.shape[:-1], "scales")
    _check(lib.jllm_kv_encode_i8(kv.data_ptr(), codes.data_ptr(), scales.data_ptr(), n, head_dim, _stream_ptr(stream)),
           "jllm_kv_encode_i8")
    return codes, scales


def jllm_kv_decode_i8(codes, scales, head_dim: int = 128, out=None, stream=None):
    """int8 codes [..., head_dim] and fp16 scales [...] -> fp16 KV vectors."""
    torch = _torch()
    if codes.shape[-1] != head_dim:
        raise ValueError("last dimension must be head_dim")
    _need(codes, torch.int8, None, "codes")
    _need(scales, torch.float16, codes.shape[:-1], "scales")
    n = codes.numel() // head_dim
    if out is None:
        out = torch.empty(codes.shape, dtype=torch.float16, device=codes.device)
    _need(out, torch.float16, codes.shape, "out")
    _check(lib.jllm_kv_decode_i8(codes.data_ptr(), scales.data_ptr(), out.data_ptr(), n, head_dim, _stream_ptr(stream)),
           "jllm_kv_decode_i8")
    return out


def jllm_q4k_ffn_swiglu(w_gate, w_up, x, N: int, K: int, out=None, ws=None, stream=None):
    """h[M, N] (fp16) = silu(X Wg^T) * (X Wu^T)."""
    torch = _torch()
    _need(w_gate, torch.uint8, _w_shape(N, K), "w_gate")
    _need(w_up, torch.uint8, _w_shape(N, K), "w_up")
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M = int(x.shape[0])
    _need(x, torch.float16, (M, K), "x")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, (M, N), "out")
    ws, nbytes = _ws(M, N, K, ws, x.device, stream)
    _check(
        lib.jllm_q4k_ffn_swiglu(w_gate.data_ptr(), w_up.data_ptr(), x.data_ptr(), out.data_ptr(), M, N, K,
                                ws.data_ptr() if ws is not None else None, nbytes, _stream_ptr(stream)),
        "jllm_q4k_ffn_swiglu",
    )
    return out

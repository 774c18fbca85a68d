"""The bounded-wait error path, exercised on the GPU without a fault.

A test build of the library (-DJLLM_FAULT_INJECTION, waits limited to 20 ms)
has a switch that makes one copy never be issued: CTA 0 of the tcgen05 GEMM
skips its first X tile, or warp 0 of CTA 0 of the GEMV skips its weight
rows.  The wait on that copy then runs out: the kernel must set its error
word, wind down (copies and MMAs in flight awaited, tensor memory freed) and
return (the GEMV chain: CTA 0's producer skips its first copy, and the other
CTAs give up waiting for CTA 0's step counter; the few-token GEMM: CTA 0 skips
its first x copies), jllm_get_device_error must report JLLM_ERR_DEVICE_TIMEOUT, and the
next calls on the same context must be correct again -- including
jllm_q4k_gemm_noalloc, whose static workspace a timed-out call leaves with
stale stream-K flags until jllm_get_device_error clears them.  Runs in a child
process so that the test library is the only one loaded there."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, sys, time
import numpy as np, torch
root, lib_path = sys.argv[1], sys.argv[2]
sys.path.insert(0, root); sys.path.insert(0, root + "/tests")
import oracle, synthetic
lib = ctypes.CDLL(lib_path)
P, I64 = ctypes.c_void_p, ctypes.c_int64
lib.jllm_q4k_gemm_noalloc.argtypes = [P, P, P, ctypes.c_int, I64, I64, I64, P]
lib.jllm_q4k_gemm.argtypes = [P, P, P, ctypes.c_int, I64, I64, I64, P, ctypes.c_size_t, P]
lib.jllm_q4k_gemv.argtypes = [P, P, P, I64, I64, P, ctypes.c_size_t, P]
lib.jllm_q4k_workspace_bytes.argtypes = [I64, I64, I64]
lib.jllm_q4k_workspace_bytes.restype = ctypes.c_size_t
lib.jllm_get_device_error.argtypes = [P]
lib.jllm_test_fault_injection.argtypes = [ctypes.c_int, ctypes.c_int]
TIMEOUT = 7
s = torch.cuda.current_stream().cuda_stream

def within(y, ref, s_):
    return bool(np.all(np.abs(y.astype(np.float64) - ref) <= oracle.tolerance(s_)))

# tcgen05 GEMM: 16 tiles of 128 tokens as clusters splitting K (no workspace), and
# 20 tiles of 256 tokens of 64 K steps with the stream-K split, whose flags a timed-out
# call leaves set (the no-alloc array: cleared by jllm_get_device_error; a caller
# workspace: zero-filled again by its owner)
for M, N, K in ((235, 1024, 2560), (300, 1280, 4096)):
    w = synthetic.q4k_weights(N, K, 9500); x = synthetic.activations(M, K, 9501)
    ref, sref = oracle.matmul(w, x, N, K)
    wd, xd = torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    noalloc = lambda: lib.jllm_q4k_gemm_noalloc(wd.data_ptr(), xd.data_ptr(), y.data_ptr(), 0, M, N, K, s)
    assert noalloc() == 0 and lib.jllm_get_device_error(s) == 0 and within(y.cpu().numpy(), ref, sref)
    for rnd in range(2):
        assert lib.jllm_test_fault_injection(1, 0) == 0
        t0 = time.time()
        assert noalloc() == 0
        st = lib.jllm_get_device_error(s)
        assert st == TIMEOUT, (M, st)
        assert time.time() - t0 < 5.0  # the kernel returned after its bounded waits
        assert lib.jllm_test_fault_injection(0, 0) == 0
        for _ in range(2):
            y.fill_(float("nan"))
            assert noalloc() == 0
            assert lib.jllm_get_device_error(s) == 0
            assert within(y.cpu().numpy(), ref, sref), ("noalloc after a timeout", M)
    need = lib.jllm_q4k_workspace_bytes(M, N, K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    gemm = lambda: lib.jllm_q4k_gemm(wd.data_ptr(), xd.data_ptr(), y.data_ptr(), 0, M, N, K, ws.data_ptr(), need, s)
    assert lib.jllm_test_fault_injection(1, 0) == 0
    assert gemm() == 0 and lib.jllm_get_device_error(s) == TIMEOUT
    assert lib.jllm_test_fault_injection(0, 0) == 0
    ws.zero_()
    assert gemm() == 0 and lib.jllm_get_device_error(s) == 0 and within(y.cpu().numpy(), ref, sref)

K = 2560
# GEMV (M = 1): warp 0 of CTA 0 never gets its rows
N1 = 4096
w1 = synthetic.q4k_weights(N1, K, 9502); x1 = synthetic.activations(1, K, 9503)
r1, s1 = oracle.matmul(w1, x1, N1, K)
w1d, x1d = torch.from_numpy(w1).cuda(), torch.from_numpy(x1.reshape(K)).cuda()
y1 = torch.empty(N1, dtype=torch.float32, device="cuda")
gemv = lambda: lib.jllm_q4k_gemv(w1d.data_ptr(), x1d.data_ptr(), y1.data_ptr(), N1, K, None, 0, s)
assert lib.jllm_test_fault_injection(0, 1) == 0
assert gemv() == 0 and lib.jllm_get_device_error(s) == TIMEOUT
assert lib.jllm_test_fault_injection(0, 0) == 0
assert gemv() == 0 and lib.jllm_get_device_error(s) == 0 and within(y1.cpu().numpy()[None, :], r1, s1)

# GEMV chain: the producer of CTA 0 never issues its first copy; the other CTAs
# then give up waiting for CTA 0's step counter
class Step(ctypes.Structure):
    _fields_ = [("count", ctypes.c_int32), ("y_f16", ctypes.c_int32), ("K", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("w_q4k", ctypes.c_void_p * 4), ("y", ctypes.c_void_p * 4),
                ("N", ctypes.c_int64 * 4)]
lib.jllm_q4k_gemv_chain.argtypes = [ctypes.POINTER(Step), ctypes.c_int, P, P]
lib.jllm_q4k_gemv_chain_sync_bytes.restype = ctypes.c_size_t
lib.jllm_test_fault_injection_chain.argtypes = [ctypes.c_int]
yc = torch.empty(N1, dtype=torch.float32, device="cuda")
steps = (Step * 3)()
for st in steps:
    st.count, st.y_f16, st.K, st.x = 1, 0, K, x1d.data_ptr()
    st.w_q4k[0], st.y[0], st.N[0] = w1d.data_ptr(), yc.data_ptr(), N1
sync = torch.zeros(lib.jllm_q4k_gemv_chain_sync_bytes(3), dtype=torch.uint8, device="cuda")
torch.cuda.synchronize()
chain = lambda: lib.jllm_q4k_gemv_chain(steps, 3, sync.data_ptr(), s)
assert chain() == 0 and lib.jllm_get_device_error(s) == 0 and within(yc.cpu().numpy()[None, :], r1, s1)
for rnd in range(2):
    assert lib.jllm_test_fault_injection_chain(1) == 0
    t0 = time.time()
    assert chain() == 0
    st_ = lib.jllm_get_device_error(s)
    assert st_ == TIMEOUT, st_
    assert time.time() - t0 < 5.0
    assert lib.jllm_test_fault_injection_chain(0) == 0
    sync.zero_()  # the caller zeroes the sync words again after a timeout
    yc.fill_(float("nan"))
    assert chain() == 0 and lib.jllm_get_device_error(s) == 0
    assert within(yc.cpu().numpy()[None, :], r1, s1), "chain after a timeout"
    assert not sync.any().item()

# few-token GEMM (warp-level tensor cores, cluster split-K): CTA 0 never issues
# its first x copies; its peers in the cluster wait for its partial sums
lib.jllm_test_fault_injection_mma.argtypes = [ctypes.c_int]
Mm, Nm = 33, 1024
wm = synthetic.q4k_weights(Nm, K, 9504); xm = synthetic.activations(Mm, K, 9505)
rm, smm = oracle.matmul(wm, xm, Nm, K)
wmd, xmd = torch.from_numpy(wm).cuda(), torch.from_numpy(xm).cuda()
ym = torch.empty((Mm, Nm), dtype=torch.float32, device="cuda")
few = lambda: lib.jllm_q4k_gemm(wmd.data_ptr(), xmd.data_ptr(), ym.data_ptr(), 0, Mm, Nm, K, None, 0, s)
assert few() == 0 and lib.jllm_get_device_error(s) == 0 and within(ym.cpu().numpy(), rm, smm)
for rnd in range(2):
    assert lib.jllm_test_fault_injection_mma(1) == 0
    t0 = time.time()
    assert few() == 0
    st_ = lib.jllm_get_device_error(s)
    assert st_ == TIMEOUT, st_
    assert time.time() - t0 < 5.0
    assert lib.jllm_test_fault_injection_mma(0) == 0
    ym.fill_(float("nan"))
    assert few() == 0 and lib.jllm_get_device_error(s) == 0
    assert within(ym.cpu().numpy(), rm, smm), "few-token GEMM after a timeout"
print("ok")
'''


def test_bounded_waits_report_timeout_and_recover():
    import importlib.util

    spec = importlib.util.spec_from_file_location("_jllm_build", os.path.join(ROOT, "bit_q4_weight_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    lib = b.build(variant="fi", extra=["-DJLLM_FAULT_INJECTION", "-DJLLM_WAIT_LIMIT_NS=20000000ull"])
    out = subprocess.run([sys.executable, "-c", CHILD, ROOT, lib], capture_output=True, text=True, timeout=900)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), (out.stdout[-2000:], out.stderr[-3000:])

"""Host-side checks of the C ABI: the library builds for sm_103a, loads, exports
every symbol include/jllm_q4k.h declares, and rejects bad arguments
synchronously without touching CUDA.  No GPU needed."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jllm_q4k.h")


@pytest.fixture(scope="module")
def q():
    import __graft_entry__

    __graft_entry__.build()
    import bit_q4_weight_gb300

    return bit_q4_weight_gb300


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jllm_\w+)\s*\(", text)))


def test_header_symbols_exported(q):
    names = _declared()
    assert set(names) == set(q.EXPORTS)
    lib = ctypes.CDLL(q.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_library_targets_sm103a(q):
    # The library is compiled for sm_103a only (one -gencode, no PTX for JIT).
    from bit_q4_weight_gb300 import _build

    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.getsize(q.LIB_PATH) > 0


def test_status_strings(q):
    for code in range(9):
        assert q.status_string(code).startswith("JLLM_")
    assert q.status_string(99) == "JLLM_ERR_UNKNOWN"


def test_workspace_and_threshold(q):
    for shape in [(1, 1024, 2560), (33, 4096, 2560), (2048, 9728, 2560), (1, 151936, 2560)]:
        assert q.jllm_q4k_workspace_bytes(*shape) >= 0
    assert q.jllm_q4k_gemv_max_m() >= 0


ALIGNED = 1 << 20  # a non-null, 16-byte-aligned fake address (never dereferenced)


@pytest.mark.parametrize(
    "args,status",
    [
        ((None, ALIGNED, ALIGNED, 0, 4, 128, 256, None, 0, None), 1),       # null W
        ((ALIGNED, ALIGNED, ALIGNED, 0, 0, 128, 256, None, 0, None), 1),    # M = 0
        ((ALIGNED, ALIGNED, ALIGNED, 0, 4, -1, 256, None, 0, None), 1),     # N < 1
        ((ALIGNED, ALIGNED, ALIGNED, 0, 4, 128, 300, None, 0, None), 2),    # K % 256
        ((ALIGNED, ALIGNED, ALIGNED, 0, 4, 128, 0, None, 0, None), 2),      # K = 0
        ((ALIGNED, ALIGNED, ALIGNED, 0, 4, 128, 1 << 40, None, 0, None), 2),  # K too large
        ((ALIGNED, ALIGNED, ALIGNED, 0, 4, (1 << 30) + 1, 256, None, 0, None), 2),  # N beyond the index range
        ((ALIGNED, ALIGNED, ALIGNED, 0, (1 << 30) + 1, 128, 256, None, 0, None), 2),  # M beyond the index range
        ((ALIGNED, ALIGNED, ALIGNED, 7, 4, 128, 256, None, 0, None), 4),    # dtype
        ((ALIGNED + 8, ALIGNED, ALIGNED, 0, 4, 128, 256, None, 0, None), 3),  # W misaligned
        ((ALIGNED, ALIGNED + 2, ALIGNED, 0, 4, 128, 256, None, 0, None), 3),  # X misaligned
        ((ALIGNED, ALIGNED, ALIGNED + 4, 1, 4, 128, 256, None, 0, None), 3),  # Y misaligned
    ],
)
def test_gemm_argument_errors(q, args, status):
    assert q.lib.jllm_q4k_gemm(*args) == status


def test_other_entry_argument_errors(q):
    A = ALIGNED
    assert q.lib.jllm_q4k_dequant(None, A, 0, 4, 256, None) == 1
    assert q.lib.jllm_q4k_dequant(A, A, 2, 4, 256, None) == 4
    assert q.lib.jllm_q4k_dequant(A, A, 0, 4, 255, None) == 2
    assert q.lib.jllm_q4k_dequant(A + 1, A, 0, 4, 256, None) == 3
    assert q.lib.jllm_q4k_gemv(A, None, A, 4, 256, None, 0, None) == 1
    assert q.lib.jllm_q4k_gemv(A, A, A, 4, 512 + 7, None, 0, None) == 2
    assert q.lib.jllm_q4k_gemv(A, A, A + 8, 4, 512, None, 0, None) == 3
    assert q.lib.jllm_q4k_ffn_swiglu(A, None, A, A, 1, 4, 256, None, 0, None) == 1
    assert q.lib.jllm_q4k_ffn_swiglu(A, A, A, A, 1, 4, 100, None, 0, None) == 2
    assert q.lib.jllm_q4k_ffn_swiglu(A, A + 4, A, A, 1, 4, 256, None, 0, None) == 3


def test_gemv_batch_argument_errors(q):
    import ctypes

    A = ALIGNED
    P = ctypes.c_void_p

    def arrs(ws, ys, ns):
        return (P * len(ws))(*ws), (P * len(ys))(*ys), (ctypes.c_int64 * len(ns))(*ns)

    w, y, n = arrs([A, A], [A, A], [4, 8])
    assert q.lib.jllm_q4k_gemv_batch(w, y, n, 0, A, 256, None) == 1  # count 0
    assert q.lib.jllm_q4k_gemv_batch(w, y, n, 9, A, 256, None) == 1  # count above 8
    assert q.lib.jllm_q4k_gemv_batch(None, y, n, 2, A, 256, None) == 1
    assert q.lib.jllm_q4k_gemv_batch(w, y, n, 2, None, 256, None) == 1
    assert q.lib.jllm_q4k_gemv_batch(w, y, n, 2, A, 300, None) == 2  # K % 256
    assert q.lib.jllm_q4k_gemv_batch(w, y, n, 2, A + 2, 256, None) == 3  # x misaligned
    w2, y2, n2 = arrs([A, None], [A, A], [4, 8])
    assert q.lib.jllm_q4k_gemv_batch(w2, y2, n2, 2, A, 256, None) == 1  # one null W
    w3, y3, n3 = arrs([A, A], [A, A + 4], [4, 8])
    assert q.lib.jllm_q4k_gemv_batch(w3, y3, n3, 2, A, 256, None) == 3  # one y misaligned
    w4, y4, n4 = arrs([A, A], [A, A], [4, 0])
    assert q.lib.jllm_q4k_gemv_batch(w4, y4, n4, 2, A, 256, None) == 1  # N < 1


def test_gemv_chain_argument_errors(q):
    A = ALIGNED
    S = q.GemvStep

    def chain(*steps):
        return (S * len(steps))(*steps)

    def step(count=2, K=2560, x=A, ws=(A, A), ys=(A, A), ns=(8, 0), f16=0):
        st = S()
        st.count, st.y_f16, st.K, st.x = count, f16, K, x
        for j in range(len(ws)):
            st.w_q4k[j], st.y[j], st.N[j] = ws[j], ys[j], ns[j]
        return st

    ok = chain(step(), step(count=1, K=12288, ws=(A,), ys=(A,), ns=(3,)))
    run = q.lib.jllm_q4k_gemv_chain
    assert run(ok, 0, A, None) == 1                       # no steps
    assert run(ok, 257, A, None) == 1                     # above the step limit
    assert run(None, 2, A, None) == 1
    assert run(ok, 2, None, None) == 1                    # no sync buffer
    assert run(ok, 2, A + 2, None) == 3                   # sync not 4-byte aligned
    assert run(chain(step(count=0)), 1, A, None) == 1
    assert run(chain(step(count=5)), 1, A, None) == 1
    assert run(chain(step(f16=2)), 1, A, None) == 1
    assert run(chain(step(x=None)), 1, A, None) == 1
    assert run(chain(step(K=300)), 1, A, None) == 2       # K % 256
    assert run(chain(step(K=12544)), 1, A, None) == 2     # K above 12288
    assert run(chain(step(x=A + 8)), 1, A, None) == 3
    assert run(chain(step(ws=(A, A + 4), ns=(8, 8))), 1, A, None) == 3
    assert run(chain(step(ws=(A, None), ns=(8, 8))), 1, A, None) == 1
    assert run(chain(step(ns=(8, -1))), 1, A, None) == 1
    assert run(chain(step(), step(K=100)), 2, A, None) == 2  # a later step is checked too
    assert q.jllm_q4k_gemv_chain_sync_bytes(0) == 0
    assert q.jllm_q4k_gemv_chain_sync_bytes(257) == 0
    assert q.jllm_q4k_gemv_chain_sync_bytes(144) == 4 * 145


def test_gemm_batch_argument_errors(q):
    import ctypes

    A = ALIGNED
    P = ctypes.c_void_p

    def arrs(ws, ys, ns):
        return (P * len(ws))(*ws), (P * len(ys))(*ys), (ctypes.c_int64 * len(ns))(*ns)

    w, y, n = arrs([A, A], [A, A], [128, 256])
    call = q.lib.jllm_q4k_gemm_batch
    assert call(w, A, y, 0, 64, n, 256, 0, None, 0, None) == 1  # count 0
    assert call(w, A, y, 0, 64, n, 256, 5, None, 0, None) == 1  # count above 4
    assert call(None, A, y, 0, 64, n, 256, 2, None, 0, None) == 1
    assert call(w, None, y, 0, 64, n, 256, 2, None, 0, None) == 1
    assert call(w, A, None, 0, 64, n, 256, 2, None, 0, None) == 1
    assert call(w, A, y, 0, 64, None, 256, 2, None, 0, None) == 1
    assert call(w, A, y, 2, 64, n, 256, 2, None, 0, None) == 4  # dtype
    assert call(w, A, y, 0, 0, n, 256, 2, None, 0, None) == 1  # M < 1
    assert call(w, A, y, 0, 64, n, 300, 2, None, 0, None) == 2  # K % 256
    assert call(w, A + 2, y, 0, 64, n, 256, 2, None, 0, None) == 3  # x misaligned
    w2, y2, n2 = arrs([A, None], [A, A], [128, 256])
    assert call(w2, A, y2, 0, 64, n2, 256, 2, None, 0, None) == 1  # one null W
    w3, y3, n3 = arrs([A, A], [A, A + 4], [128, 256])
    assert call(w3, A, y3, 0, 64, n3, 256, 2, None, 0, None) == 3  # one y misaligned
    w4, y4, n4 = arrs([A, A], [A, A], [128, 0])
    assert call(w4, A, y4, 0, 64, n4, 256, 2, None, 0, None) == 1  # N < 1


def test_gemv_rmsnorm_batch_argument_errors(q):
    import ctypes

    A = ALIGNED
    P = ctypes.c_void_p
    w = (P * 2)(A, A)
    y = (P * 2)(A, A)
    n = (ctypes.c_int64 * 2)(4, 8)
    call = q.lib.jllm_q4k_gemv_rmsnorm_batch
    assert call(w, y, n, 2, A, None, 1e-6, 256, None) == 1  # no gamma
    assert call(w, y, n, 0, A, A, 1e-6, 256, None) == 1  # count 0
    assert call(w, y, n, 9, A, A, 1e-6, 256, None) == 1  # count above 8
    assert call(w, y, n, 2, A, A, -1.0, 256, None) == 1  # eps < 0
    assert call(w, y, n, 2, A, A, float("nan"), 256, None) == 1  # eps NaN
    assert call(w, y, n, 2, A, A + 4, 1e-6, 256, None) == 3  # gamma misaligned
    assert call(w, y, n, 2, A + 2, A, 1e-6, 256, None) == 3  # x misaligned
    assert call(w, y, n, 2, A, A, 1e-6, 300, None) == 2  # K % 256


def _no_cuda():
    try:
        import torch

        return not torch.cuda.is_available()
    except Exception:
        return True


@pytest.mark.skipif(not _no_cuda(), reason="only meaningful where no CUDA device exists")
def test_valid_call_without_device_reports_error(q):
    # With valid arguments and no device the call must fail cleanly, never crash.
    st = q.lib.jllm_q4k_gemm(ALIGNED, ALIGNED, ALIGNED, 0, 4, 128, 256, None, 0, None)
    assert st in (q.JLLM_ERR_CUDA, q.JLLM_ERR_NO_DEVICE)


def test_python_wrappers_validate_tensors(q):
    torch = pytest.importorskip("torch")
    w = torch.zeros((4, 144), dtype=torch.uint8)
    x = torch.zeros((1, 256), dtype=torch.float16)
    with pytest.raises(ValueError):
        q.jllm_q4k_gemm(w, x, 4, 256)  # CPU tensors are rejected before any call

"""The int8 tensor-core question for this part, answered by the toolchain: the
CUDA assembler refuses tcgen05.mma .kind::i8 for sm_103a, so an int8 ("MMQ")
prefill variant has no 5th-generation tensor-core instruction to run on (the
warp-level mma.sync s8 rate is measured by bench.py --tc-rates).  CPU only:
nvcc cross-compiles, nothing runs."""
import os
import shutil
import subprocess

import pytest

SRC = r'''
__global__ void k(unsigned d, unsigned long long a, unsigned long long b, unsigned idesc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::KIND [%0], %1, %2, %3, p;\n}" ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(1));
}
'''


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    pytest.skip("nvcc not available")


@pytest.mark.parametrize("kind,ok", [("f16", True), ("i8", False)])
def test_tcgen05_kinds_on_sm103a(tmp_path, kind, ok):
    src = tmp_path / "k.cu"
    src.write_text(SRC.replace("KIND", kind))
    res = subprocess.run([_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-c", str(src), "-o",
                          str(tmp_path / "k.o")], capture_output=True, text=True)
    if ok:
        assert res.returncode == 0, res.stderr
    else:
        assert res.returncode != 0
        assert "kind::i8" in res.stderr and "not supported" in res.stderr and "sm_103a" in res.stderr

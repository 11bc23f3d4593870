"""GPU: the C boundary called from a C program (no Python, no PyTorch on the
path): one append + decode step, one few-queries verification step, the
same rows through pa_prefill, the page scores and two block copies on
cudaMalloc'd memory, checked against the oracle inside the program
(tests/c_abi/decode_from_c.c)."""

import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_step_from_c(tmp_path):
    import __graft_entry__
    import oracle
    __graft_entry__.build()
    lib_dir = os.path.join(ROOT, "paged_kv_cache_202_gb300")
    ora = oracle.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cc = shutil.which("gcc") or "gcc"
    exe = str(tmp_path / "decode_from_c")
    subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-o", exe,
                    os.path.join(ROOT, "tests", "c_abi", "decode_from_c.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", lib_dir, "-lpa", "-L", os.path.dirname(ora), "-loracle",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.dirname(ora)}",
                    f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr

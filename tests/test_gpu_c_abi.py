"""The C ABI from plain C: tests/c_abi/ring_thc.c is compiled with gcc
against include/gar.h, libgar.so and the CUDA runtime (no Python or PyTorch
in the program) and run on the GPU; it checks the ring average exactly, a
uniform and a non-uniform THC round within their quantization intervals and
an RHT round trip within the transform's error bound."""
import glob
import os
import shutil
import subprocess

import pytest

from helpers import need_cuda

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_lib_dir():
    for d in ["/usr/local/cuda/lib64"] + glob.glob("/usr/local/cuda/targets/*/lib"):
        if glob.glob(os.path.join(d, "libcudart.so*")):
            return d
    pytest.skip("libcudart not found")


def test_plain_c_program(tmp_path):
    need_cuda()  # builds libgar.so and checks for a GPU
    import gradient_allreduce_homomorphic_gb300 as g

    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(g.LIB_PATH)
    cuda_lib = _cuda_lib_dir()
    exe = str(tmp_path / "ring_thc")
    subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", "/usr/local/cuda/include", os.path.join(ROOT, "tests", "c_abi", "ring_thc.c"),
                    "-o", exe, "-L", lib_dir, "-lgar", "-L", cuda_lib, "-lcudart", "-lm",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cuda_lib}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("c abi ok"), r.stdout

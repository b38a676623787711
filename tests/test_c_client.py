"""A plain C program uses the C ABI: it includes include/slide.h, links
libslide.so and the CUDA runtime, and calls the entry points directly (no
Python, no torch).  Host-only calls run without a GPU; the GPU part checks a
closed form (zero gradients from zero moments: pure decay) with device and
with host gradient buffers, and that a refused call changes nothing."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_client.c")


def _build(tmp_path):
    from mixed_precision_adam_grad_gb300 import build
    lib = build.build()
    exe = str(tmp_path / "abi_client")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cuda_lib = os.path.join(cuda, "lib64")
    subprocess.run(["gcc", "-std=c99", "-O1", "-Wall", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), SRC, "-o", exe,
                    "-L", os.path.dirname(lib), "-lslide", f"-Wl,-rpath,{os.path.dirname(lib)}",
                    "-L", cuda_lib, "-lcudart", f"-Wl,-rpath,{cuda_lib}"], check=True)
    return exe


def test_c_client_host_calls(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe, "cpu"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_c_client_gpu_step(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _build(tmp_path)
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

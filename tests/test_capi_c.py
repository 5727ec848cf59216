"""The C ABI used from a C program (CPU only): tests/c/capi_host.c is built
with gcc -std=c99 against include/latentmoe.h and the in-tree library, then
run; it checks the host-side answers of the entry points."""
import os
import shutil
import subprocess

import pytest

from mixture_experts_layer_router_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_compiles_as_c_and_host_checks_hold(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = build.build()
    exe = str(tmp_path / "capi_host")
    libdir = os.path.dirname(lib)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-o", exe,
                        os.path.join(ROOT, "tests", "c", "capi_host.c"),
                        "-I", os.path.join(ROOT, "include"), "-L", libdir, "-llatentmoe",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.mark.gpu
def test_forward_from_c(tmp_path):
    """tests/c/capi_forward.c: create, load seeded weights, two forwards, status,
    destroy, all from C with the CUDA runtime for device memory."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = build.build()
    libdir = os.path.dirname(lib)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cuda_lib = next((p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                 os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                                 os.path.join(cuda, "targets", "x86_64-linux", "lib"))
                     if os.path.exists(os.path.join(p, "libcudart.so"))), None)
    if cuda_lib is None:
        pytest.skip("no libcudart.so")
    exe = str(tmp_path / "capi_forward")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2", "-o", exe,
                        os.path.join(ROOT, "tests", "c", "capi_forward.c"),
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                        "-L", libdir, "-llatentmoe", "-L", cuda_lib, "-lcudart", "-lm",
                        f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cuda_lib}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr

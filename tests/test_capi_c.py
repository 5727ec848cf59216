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

"""The C ABI from C: include/mse.h compiles as C99 with -Wall -Werror, and a C program
linked against libmse.so calls its host-only entry points (no GPU involved)."""
import os
import shutil
import subprocess

import pytest

from moe_shared_expert_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gpu_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
@pytest.mark.skipif(_gpu_visible(), reason="its validation call uses non-device pointers; run without a GPU")
def test_header_is_c99_and_library_links_from_c(tmp_path):
    lib = _build.build()
    exe = tmp_path / "abi_check"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", str(exe), lib,
           "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.stdout, r.stderr)
    assert r.stdout.startswith("mse ")

"""The C ABI from plain C: tests/c_abi_host.c is compiled as C99 against
include/oomb.h, linked to liboomb.so and run (host-side paths only, no GPU)."""
import os
import shutil
import subprocess

import pytest

from paged_sparse_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c99_consumer_links_and_runs():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = build.build()
    out_dir = os.path.join(build.BUILD, "c_abi_host")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "c_abi_host")
    cuda_lib = [p for p in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
                            "/usr/local/cuda/targets/x86_64-linux/lib") if os.path.isdir(p)]
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_host.c"), "-o", exe, "-L", os.path.dirname(lib), "-loomb",
           "-Wl,-rpath," + os.path.dirname(lib)]
    for p in cuda_lib:
        cmd += ["-Wl,-rpath-link," + p, "-Wl,-rpath," + p]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout

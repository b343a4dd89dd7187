"""The backward's host-side work-split policy (tests/bwd_split_host.cpp), linked
against the library's object files and run on the host: it picks the CTA counts
that measured fastest on the benchmark's workload shapes."""
import glob
import os
import shutil
import subprocess

import pytest

from paged_sparse_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_split_policy_on_benchmark_shapes():
    nvcc = build._nvcc()
    if shutil.which(nvcc) is None and not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    build.build()
    objs = sorted(glob.glob(os.path.join(build.BUILD, "*.o")))
    out_dir = os.path.join(build.BUILD, "bwd_split_host")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "bwd_split_host")
    cmd = [nvcc, *build.ARCH, "-std=c++17", os.path.join(ROOT, "tests", "bwd_split_host.cpp"), *objs, "-o", exe,
           "-lcuda", "-lcudart", "-lcublasLt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "cannot find -lcuda" in r.stderr:
        cmd.remove("-lcuda")
        r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr

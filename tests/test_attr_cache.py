"""Host test of the per-device kernel-attribute cache the launchers use.

The dynamic shared-memory limit of a kernel is a per-device attribute: a
process that drives several GPUs must set it on each.  The cache
(``csrc/attr_cache.h``) is plain C++ with the CUDA call passed in, so this
test compiles it with the host compiler against a fake setter and runs it,
including from 16 threads at once.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "mla_latent_kv_12_gb300", "csrc")


def test_attr_cache_sets_once_per_kernel_and_device(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "attr_cache_test"
    subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, os.path.join(HERE, "attr_cache_test.cpp"),
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"

"""The per-context setting cache the library keys its launch attributes on
(csrc/vc_ctx_cache.h), checked on the host: built with g++ from
ctx_cache_check.cpp and run.  Covers the same context (recorded), a larger
size (applied again), another device, a new context after a device reset,
another kernel, a failed setting (not recorded), a key the setting completes,
and eight host threads racing on four contexts (one setting per context)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ctx_cache(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "ctx_cache_check")
    src = os.path.join(ROOT, "tests", "ctx_cache_check.cpp")
    inc = os.path.join(ROOT, "bit_fp8_attention_means_gb300", "csrc")
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", inc, src, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr

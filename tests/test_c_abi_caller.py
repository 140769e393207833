"""The C ABI from a plain C program: tests/c_abi/host_calls.c is compiled
with gcc against include/pagedkv.h only (no CUDA or PyTorch headers), linked
with libpagedkv.so and run on the host (allocator, scheduler, argument
validation; no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from paged_kv_cache_220_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_caller(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    lib = build.build()
    exe = str(tmp_path / "host_calls")
    src = os.path.join(ROOT, "tests", "c_abi", "host_calls.c")
    r = subprocess.run(["gcc", "-std=c11", "-O1", "-Wall", "-Werror", "-I",
                        os.path.join(ROOT, "include"), src, "-o", exe,
                        "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
                        "-Wl,-rpath," + os.path.dirname(lib)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr

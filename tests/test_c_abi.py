"""The C ABI from a plain C program (no PyTorch, no GPU): include/pkv.h
compiles as C and the host-only entry points of libpkv.so work."""

import os
import shutil
import subprocess

import pytest

from paged_kv_attention_17_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_host(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = pkv_build.build()
    exe = tmp_path / "abi_check"
    src = os.path.join(ROOT, "tests", "c", "abi_check.c")
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        src, "-o", str(exe), os.path.abspath(lib),
                        "-Wl,-rpath," + os.path.dirname(os.path.abspath(lib))],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "abi ok", r.stdout + r.stderr

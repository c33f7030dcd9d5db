"""The C ABI from C: tests/c_abi_check.c is compiled with the system C
compiler against include/kdkl.h, linked to the in-tree libkdkl.so and run.
No GPU and no Python binding are involved in what it checks."""
import os
import shutil
import subprocess

import pytest

from lm_head_top_gb300 import kdkl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_links_and_passes():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(kdkl.LIB_PATH):
        from lm_head_top_gb300 import build
        build.build()
    libdir = os.path.dirname(kdkl.LIB_PATH)
    out = os.path.join(ROOT, "_build")  # the in-tree build folder (not versioned)
    os.makedirs(out, exist_ok=True)
    exe = os.path.join(out, "c_abi_check")
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", libdir, "-lkdkl",
           "-Wl,-rpath," + libdir, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr

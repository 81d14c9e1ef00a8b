"""The C ABI used from plain C99: include/attn.h compiles as C, the shared library links, and
validation answers through the C calling convention (no device needed, nothing is launched)."""
import os
import shutil
import subprocess

import pytest

from attention_attn_prefill_02_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_c99_program_against_the_header(tmp_path):
    lib = binding._build.build_library()
    exe = tmp_path / "abi_check"
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi", "abi_check.c"),
           "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_check: ok" in r.stdout

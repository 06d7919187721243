"""The boundary from C: tests/c_consumer.c compiles against include/spectree.h
with a C compiler, links libspectree.so, and runs on the CPU (it calls only
host entry points and argument checks)."""
import os
import shutil
import subprocess

import pytest

from tree_speculative_verification_spec_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_uses_the_library(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = build.build()
    exe = str(tmp_path / "c_consumer")
    subprocess.check_call([cc, "-std=c11", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c_consumer.c"), lib, "-o", exe,
                           "-Wl,-rpath," + os.path.dirname(lib)])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "c consumer: ok" in out.stdout

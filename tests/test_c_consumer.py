"""The C ABI from a plain C99 program (tests/c/consumer.c): include/mxq.h
compiles as strict C, the program links against libmxq.so and its queries
and argument checks behave as documented without a GPU."""

import os
import shutil
import subprocess

import pytest

from conftest import ROOT


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c99_program_uses_the_abi(tmp_path):
    from mxfp8_block_scaled_inv_gb300 import build as B

    lib = B.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "consumer")
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "consumer.c"),
                    "-L", libdir, "-lmxq", "-Wl,-rpath," + libdir, "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "0 failures"

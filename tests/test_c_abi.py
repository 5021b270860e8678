"""A plain C11 program (tests/csrc/abi_check.c) compiles against
include/fp8bs.h, links every entry point of libfp8bs.so (no undefined
symbols allowed) and checks the validation status of each call through the
C calling convention.  No GPU: every call it makes is refused before the
library touches CUDA."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None or
                                (shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc")),
                                reason="gcc or nvcc not available")


def test_c_client_compiles_links_and_validates(tmp_path):
    from fp8_block_scaled_02_gb300 import build
    lib = build.build()
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                    os.path.join(ROOT, "tests", "csrc", "abi_check.c"),
                    lib, "-Wl,--no-undefined", "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    words = out.stdout.split()
    assert words[-4] == "checks" and int(words[-3]) > 60 and words[-2] == "failures" and words[-1] == "0", out.stdout

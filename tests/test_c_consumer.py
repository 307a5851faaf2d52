"""include/prism.h is plain C: a C99 program (tests/c/abi_consumer.c) compiles against it
with gcc -std=c99 -pedantic, links libprism.so and gets the documented answers from the
host-side parts of the ABI (CPU only)."""
import os
import shutil
import subprocess

import pytest

from linear_recurrent_sequence_causal_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c99_program_uses_the_abi(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = build.build()
    exe = tmp_path / "abi_consumer"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_consumer.c"),
           "-o", str(exe), "-L", os.path.dirname(lib), "-lprism", "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr

"""The C ABI from C: tests/c/abi_from_c.c includes include/tnd_attn.h as C99
with every warning an error, links against the built library and runs its
first-phase, status, option and plan checks (no GPU needed)."""

import os
import subprocess

import pytest

from attention_backward_tnd_b300 import build as tbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_dir():
    tbuild.build()
    return os.path.join(ROOT, "attention_backward_tnd_b300")


def test_header_compiles_as_c99_and_calls_work(lib_dir, tmp_path):
    exe = str(tmp_path / "abi_from_c")
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Wpedantic", "-Werror",
                           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
                           "-L", lib_dir, "-ltndattn", f"-Wl,-rpath,{lib_dir}", "-o", exe])
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr

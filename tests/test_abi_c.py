"""The C ABI used from C: a C11 program that includes only ``include/gqa_attn.h``
and links ``libgqa_attn.so`` compiles with -Wall -Werror and runs (no GPU needed:
it only exercises the size helpers and the host-side argument checks)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_compiles_as_c_and_program_runs(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    from gqa_attention_gb300 import build

    lib = build.build()
    exe = tmp_path / "abi_smoke"
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_smoke.c"), lib,
                           "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "abi_smoke: ok" in out.stdout

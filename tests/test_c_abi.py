"""The C ABI from a plain C99 program: include/qmoe.h compiles with gcc -std=c99
-Wall -Werror, links against libqmoe.so, and the host-only calls behave as the
header states (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

from quantized_moe_grouped_route_gb300 import qmoe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_compiles_as_c99_and_host_calls_work(tmp_path):
    qmoe.lib()  # built in-tree
    libdir = os.path.dirname(qmoe.LIB_PATH)
    exe = str(tmp_path / "abi_from_c")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                    os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
                    "-o", exe, "-L", libdir, "-lqmoe", "-Wl,-rpath," + libdir, "-lm"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok: 0 failure(s)" in r.stdout

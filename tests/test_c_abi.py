"""The C ABI from plain C: ``tests/c_abi_host_checks.c`` includes only
``include/pkv.h`` (no CUDA, C++ or Python headers), is compiled as strict C11
with warnings as errors, links against ``libpkv.so`` and runs its host-side
checks. CPU only: every call in it is a size query or is rejected by the
library's argument checks before any CUDA runtime call."""

import os
import shutil
import subprocess

import pytest

from paged_kv_decode_05_gb300.build import LIB, build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_header_compiles_as_c_and_host_checks_pass(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    build()
    exe = str(tmp_path / "c_abi_host_checks")
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(HERE, "c_abi_host_checks.c"), "-o", exe,
                    "-L", os.path.dirname(LIB), "-lpkv",
                    "-Wl,-rpath," + os.path.dirname(LIB)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"

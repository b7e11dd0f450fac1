"""A C host program compiled against include/mqa.h and linked with libmqa.so:
the header is valid C, every call links, and host-side validation answers
through the plain C ABI (no Python in between, no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from fp8_mqa_indexer_gb300 import build as mqa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_compiles_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler on this host")
    lib = mqa_build.build()
    exe = str(tmp_path / "abi_check")
    src = os.path.join(ROOT, "tests", "c", "abi_check.c")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                        "-o", exe, "-L", os.path.dirname(lib), "-lmqa",
                        "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_check: ok" in r.stdout

"""The C ABI from plain C: tests/c/abi_from_c.c compiled as C99 against
include/mfsdp.h alone and linked to the shared library (no torch, no C++), run
on the host.  It exercises the planner, the size queries, the group query, the
host-side argument checks and the status strings."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_abi_from_plain_c(mfsdp, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(mfsdp.library_path())
    exe = str(tmp_path / "abi_from_c")
    build = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                            os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-o", exe, "-L", lib_dir, "-lmfsdp",
                            "-Wl,-rpath," + lib_dir], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.startswith("ok " + mfsdp.version())

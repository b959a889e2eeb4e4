"""The C ABI from plain C: tests/c/abi_from_c.c compiled as C99 against
include/mfsdp.h alone and linked to the shared library (no torch, no C++), run
on the host.  It exercises the planner, the size queries, the group query, the
host-side argument checks, an owner-shard checkpoint and the status strings."""
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
    run = subprocess.run([exe, str(tmp_path / "rank0.ck")], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.startswith("ok " + mfsdp.version())
    ck = mfsdp.checkpoint_load(str(tmp_path / "rank0.ck"))      # the C program's file, read back here
    assert (ck.header.world, ck.header.rank, ck.header.adam_step) == (2, 1, 3)
    assert ck.momentum[10] == 10 * 0.5 - 7.0


@pytest.mark.gpu
def test_owner_step_from_plain_c(mfsdp, tmp_path):
    """tests/c/step_from_c.c: an owner step with device memory from cudaMalloc
    and no framework, through the workspace and the no-workspace entry points."""
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if not cc or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("no C compiler or CUDA headers")
    lib_dir = os.path.dirname(mfsdp.library_path())
    exe = str(tmp_path / "step_from_c")
    cuda_lib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                     if os.path.exists(os.path.join(d, "libcudart.so"))), os.path.join(cuda, "lib64"))
    build = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                            "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "step_from_c.c"),
                            "-o", exe, "-L", lib_dir, "-lmfsdp", "-L", cuda_lib, "-lcudart", "-lm",
                            "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + cuda_lib], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    if run.returncode == 2:
        pytest.skip("no CUDA device")
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("ok"), run.stdout

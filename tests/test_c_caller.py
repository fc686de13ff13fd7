"""The C ABI from C: tests/ra_c_caller.c, compiled with the system C compiler
against include/ra.h and linked to libra.so and the CUDA runtime, runs its host
checks (chunk bounds of the tirogla.com self-test shape, argument errors caught
before any launch) without a GPU, and its device checks (the same page's
closed form 5*i + 10030 through all-reduce, reduce-scatter and all-gather, and
the fp32 average on a created stream) on one."""

import glob
import os
import shutil
import subprocess

import pytest
import torch

from conftest import ROOT


@pytest.fixture(scope="module")
def caller(tmp_path_factory):
    from ring_all_reduce_02_gb300 import build

    build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(build._nvcc())))
    libdir = os.path.dirname(build.LIB)
    dirs = [os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")] + glob.glob(os.path.join(cuda, "targets", "*", "lib"))
    cudalib = next((d for d in dirs if os.path.exists(os.path.join(d, "libcudart.so"))), None)
    if cudalib is None:
        pytest.skip("no shared CUDA runtime to link the C caller against")
    exe = str(tmp_path_factory.mktemp("c_caller") / "ra_c_caller")
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Werror", f"-I{os.path.join(ROOT, 'include')}",
           f"-I{os.path.join(cuda, 'include')}", os.path.join(ROOT, "tests", "ra_c_caller.c"), "-o", exe,
           f"-L{libdir}", "-lra", f"-Wl,-rpath,{libdir}", f"-L{cudalib}", "-lcudart", f"-Wl,-rpath,{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_caller_host_checks(caller):
    r = subprocess.run([caller, "--host-only"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "C ABI HOST OK" in r.stdout, r.stdout + r.stderr


@pytest.mark.gpu
def test_c_caller_device_checks(caller):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    r = subprocess.run([caller], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "C ABI OK" in r.stdout, r.stdout + r.stderr

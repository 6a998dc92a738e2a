"""The C ABI driven from plain C: tests/c_abi/abi_check.c includes include/hsi.h
as C11, links against libhsi.so and checks the documented behaviour (host
argument checks here; one hsi_topk on the device in the GPU test)."""
import os
import shutil
import subprocess

import pytest

import long_context_decode_lightning_gb300 as hsi
from conftest import ROOT

needs_tools = pytest.mark.skipif(shutil.which("nvcc") is None or shutil.which("gcc") is None,
                                 reason="nvcc or gcc not on PATH")


def _cuda_home():
    return os.path.dirname(os.path.dirname(os.path.realpath(shutil.which("nvcc"))))


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    so = hsi.build()
    out = str(tmp_path_factory.mktemp("c_abi") / "abi_check")
    cuda = _cuda_home()
    libdir = os.path.join(cuda, "lib64")
    if not os.path.isdir(libdir):
        libdir = os.path.join(cuda, "lib")
    subprocess.check_call([
        "gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O1",
        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
        os.path.join(ROOT, "tests", "c_abi", "abi_check.c"), "-o", out,
        "-L", os.path.dirname(so), "-lhsi", "-Wl,-rpath," + os.path.dirname(so),
        "-L", libdir, "-lcudart", "-Wl,-rpath," + libdir])
    return out


@needs_tools
def test_c_program_host_checks(exe):
    r = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr


@needs_tools
@pytest.mark.gpu
def test_c_program_topk_on_device(exe):
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr

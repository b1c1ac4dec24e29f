"""The C ABI used from a plain C program (tests/c_abi/decode_step.c): the
decode step's cache write, GQA decode with and without splits and absorbed
MLA decode on cudaMalloc'd buffers, checked against closed forms.  On the
CPU the program is only compiled (C11, warnings as errors) and linked."""
import os
import subprocess

import pytest

from gqa_mqa_mla_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def compile_decode_step(exe: str) -> None:
    lib = build.build()
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(build._nvcc())))
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-Wall", "-Wextra", "-Werror",
                           os.path.join(HERE, "c_abi", "decode_step.c"),
                           f"-I{os.path.join(ROOT, 'include')}",
                           f"-I{os.path.join(cuda, 'include')}", "-o", exe, lib,
                           f"-L{os.path.join(cuda, 'lib64')}", "-lcudart", "-lm",
                           f"-Wl,-rpath,{os.path.dirname(lib)}",
                           f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"])


def test_decode_step_compiles_as_c(tmp_path):
    exe = str(tmp_path / "decode_step")
    compile_decode_step(exe)
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_decode_step_from_c(tmp_path):
    exe = str(tmp_path / "decode_step")
    compile_decode_step(exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout

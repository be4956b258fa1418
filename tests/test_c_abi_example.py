"""The C ABI from plain C: tests/c_abi_example.c compiles with gcc against
include/msda.h and links libmsda.so and the CUDA runtime (CPU); on a GPU it
runs and checks a closed-form result (constant map)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "scale_deformable_attention_06_b300")
CUDA = "/usr/local/cuda"


def _build(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    exe = str(tmp_path / "c_abi_example")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_abi_example.c"), "-o", exe,
           "-L", PKG, "-lmsda_link", "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + PKG + "," + "-rpath," + os.path.join(CUDA, "lib64")]
    # link against the in-tree library by its file name
    cmd[cmd.index("-lmsda_link")] = os.path.join(PKG, "libmsda.so")
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_consumer_compiles_and_links(tmp_path):
    exe = _build(tmp_path)
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_c_consumer_runs(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad call rejected: 1" in r.stdout

"""The C ABI from a plain C program (tests/c/abi_demo.c), without Python in the loop."""
import os
import subprocess

import pytest

import fully_sharded_gb300 as fs
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def demo(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("c") / "abi_demo")
    lib_dir = os.path.dirname(fs.library_path())
    ora_dir = os.path.dirname(oracle.build())
    cmd = ["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c", "abi_demo.c"), "-o", out,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-l:libfsdp_gb300.so", "-L", ora_dir, "-l:libfsdp_oracle.so",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + ora_dir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("cannot build the C demo here: " + r.stderr[-300:])
    return out


def test_host_calls_from_c(demo):
    r = subprocess.run([demo, "host"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_fused_step_from_c_matches_oracle(demo):
    r = subprocess.run([demo, "gpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bit for bit" in r.stdout

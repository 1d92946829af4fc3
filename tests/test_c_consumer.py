"""The C ABI from plain C: tests/c_consumer.c is compiled with gcc against
include/mla.h and the built library (no Python, no PyTorch in the program)
and run.  Host mode needs no GPU; GPU mode runs one append + decode through
cudaMalloc'd buffers and checks a closed form (one cached token: out_h =
W^UV_h c_0)."""
import os
import shutil
import subprocess

import pytest

from mla_decode_attention_paged_gb300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    mla_build.build()
    libdir = os.path.dirname(mla_build.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_consumer") / "c_consumer")
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_consumer.c"), "-L", libdir, "-lmla_gb300",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm", f"-Wl,-rpath,{libdir}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_consumer_host_calls(consumer):
    r = subprocess.run([consumer, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr


@pytest.mark.gpu
def test_c_consumer_decode_on_gpu(consumer):
    r = subprocess.run([consumer, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr

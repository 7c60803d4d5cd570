"""Host time of one wq_matmul call, measured from C (tests/host_cost.c, linked
against libwq.so and the CUDA runtime): the library's own validation,
cached plan and tensor-map lookups and the launch, without Python or ctypes.
The bound is loose (a launch costs a few microseconds); the figure itself is
printed for the record."""
import json
import os
import shutil
import subprocess

import pytest

from weight_only_quantized_wq_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    lib = build.build()
    out = str(tmp_path_factory.mktemp("hc") / "host_cost")
    cuda = os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"))
    subprocess.check_call(["gcc", "-O2", "-o", out, os.path.join(HERE, "host_cost.c"), "-I" + build.INCLUDE,
                           "-I" + os.path.join(cuda, "include"), "-L" + os.path.dirname(lib), "-lwq",
                           "-L" + os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.dirname(lib),
                           "-Wl,-rpath," + os.path.join(cuda, "lib64")])
    return out


@pytest.mark.parametrize("M,K,N", [(16, 8192, 28672), (1, 4096, 11008), (1024, 8192, 28672)])
def test_host_cost_per_call(exe, M, K, N):
    r = subprocess.run([exe, str(M), str(K), str(N), "200"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    print("host cost", d)
    assert d["host_us_min"] < 50.0

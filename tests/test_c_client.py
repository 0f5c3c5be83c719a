"""The C ABI from plain C: tests/c_client/kvx_c_client.c, built with gcc as C99.

The CPU test compiles it with -std=c99 -pedantic -Werror against include/kvx.h,
links it against libkvx.so, the C oracle and the CUDA runtime, and runs the
entry points that need no GPU. The GPU test runs its three-hop chain (H2D, D2D
through a reusable descriptor buffer, D2H) on device 0, checked whole-pool
against the oracle inside the program.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "kvx_c_client.c")


def _cuda_root():
    from expert_host_block_gb300 import build as B
    return os.path.dirname(os.path.dirname(os.path.realpath(B.nvcc())))


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.fail("gcc is needed to build the C client")
    import oracle
    from expert_host_block_gb300 import build as B
    kvx_lib = B.build()
    oracle_lib = oracle.build()
    cuda = _cuda_root()
    out = str(tmp_path_factory.mktemp("c_client") / "kvx_c_client")
    libdirs = [os.path.dirname(kvx_lib), os.path.dirname(oracle_lib), os.path.join(cuda, "lib64")]
    cmd = (["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O2",
            "-I" + os.path.join(ROOT, "include"), "-isystem", os.path.join(cuda, "include"), SRC, "-o", out]
           + [f"-L{d}" for d in libdirs] + ["-lkvx", "-loracle", "-lcudart"]
           + [f"-Wl,-rpath,{d}" for d in libdirs])
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, " ".join(cmd) + "\n" + r.stdout + r.stderr
    return out


def test_c_client_builds_as_c99_and_runs_host_entry_points(client):
    r = subprocess.run([client, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("c client ok"), r.stdout + r.stderr


@pytest.mark.gpu
def test_c_client_three_hops_on_the_gpu(client):
    r = subprocess.run([client, "copy"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "c client ok" in r.stdout and "bit-exact" in r.stdout, r.stdout + r.stderr

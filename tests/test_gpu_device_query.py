"""The bulk copy path leaves the per-thread stack limit and device memory alone.

On sm_120 the cluster-scope destination form of the bulk copy made the driver raise
the per-thread stack limit on first launch and hold 1.37 GiB of device memory
(FreeToken issue #751, §What we changed). kvx issues the .shared::cta form;
this checks, in a fresh process, that the first bulk launch changes neither.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, %r)
from expert_host_block_gb300 import kvx
torch.cuda.set_device(0)
src = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
dst = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
torch.cuda.synchronize()
before = kvx.kvx_device_query()
s = src.data_ptr() + 16384 * np.arange(4096, dtype=np.uint64)
d = dst.data_ptr() + 16384 * np.arange(4096, dtype=np.uint64)
kvx.kvx_copy_batch_ex(s, d, np.full(4096, 16384), None, "d2d", {"variant": "bulk", "stages": 12}, None)
kvx.kvx_stream_check(None)
after = kvx.kvx_device_query()
print(before["stack_bytes_per_thread"], after["stack_bytes_per_thread"], before["free_bytes"], after["free_bytes"],
      after["sm_count"])
""" % ROOT


def test_bulk_launch_leaves_stack_limit_and_memory():
    out = subprocess.run([sys.executable, "-c", SCRIPT], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr
    st0, st1, f0, f1, sms = (int(x) for x in out.stdout.split())
    assert st1 == st0
    assert f0 - f1 < 64 << 20, f"free device memory fell by {(f0 - f1) >> 20} MiB"
    assert sms >= 1

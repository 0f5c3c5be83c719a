"""Destroyed descriptor buffers and device lists are argument errors, not a use after free.

The host-side fault injection of a destroyed descriptor buffer: every entry
point that takes a kvx_desc_buf or kvx_devlist looks it up in the library's
registry of live handles first, so a handle used after kvx_*_destroy (or
destroyed twice) returns KVX_ERR_INVALID_ARG and enqueues nothing, while live
handles created afterwards keep working and copy bit-exactly.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _rejected(call):
    with pytest.raises(kvx.KvxError) as e:
        call()
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG and "not a live" in str(e.value)


def test_destroyed_desc_buf_and_devlist_are_rejected():
    stale = kvx.kvx_desc_buf_create(64)
    kvx.kvx_desc_buf_destroy(stale)
    _rejected(lambda: kvx.kvx_desc_buf_info(stale))
    _rejected(lambda: kvx.kvx_upload_descriptors(stale, [8], [16], [8], None, "d2d"))
    _rejected(lambda: kvx.kvx_copy_uploaded(stale))
    _rejected(lambda: kvx.kvx_copy_uploaded_ex(stale, {"variant": "ldg"}))
    _rejected(lambda: kvx.kvx_desc_buf_destroy(stale))
    lst = kvx.kvx_devlist_create(16)
    kvx.kvx_devlist_destroy(lst)
    _rejected(lambda: kvx.kvx_copy_device_list(lst, 8, 8, 8, 4, "d2d"))
    _rejected(lambda: kvx.kvx_devlist_destroy(lst))
    kvx.kvx_stream_check(None)  # nothing was enqueued, nothing reported


def test_live_buffers_still_copy_after_stale_ones_were_rejected():
    specs = {"src": W.PoolSpec("src", "device", 8 * W.MIB, "random", (98,)),
             "dst": W.PoolSpec("dst", "device", 8 * W.MIB, "canary")}
    p = Pools(specs)
    try:
        g = np.random.default_rng([W.SEED, 98])
        n = 512
        so = (g.permutation(512)[:n] * 16384 + 8 * g.integers(0, 2, n)).astype(np.uint64)
        do = (g.permutation(512)[:n] * 16384 + 8 * g.integers(0, 2, n)).astype(np.uint64)
        sz = (8 * g.integers(1, 2047, n)).astype(np.uint64)
        b = W.Batch("src", "dst", so, do, sz, "d2d")
        want = {name: p.snapshot(name) for name in p.specs}
        src = want["src"].copy()
        oracle.copy_batch(want["dst"], src, so + np.uint64(W.GUARD), do + np.uint64(W.GUARD), sz)
        for _ in range(3):  # handles are created and destroyed around the live one
            kvx.kvx_desc_buf_destroy(kvx.kvx_desc_buf_create(n))
        with kvx.DescBuf(n) as buf:
            gone = kvx.kvx_desc_buf_create(n)
            kvx.kvx_desc_buf_destroy(gone)
            _rejected(lambda: kvx.kvx_copy_uploaded(gone))
            buf.upload(*p.addrs(b), "d2d")
            buf.copy()
            kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()

"""The batch at the chunk-count limit: KVX_MAX_CHUNKS descriptors in one call, bit-exact.

4,194,304 shuffled 8-byte descriptors (one chunk each, so the chunk table holds
exactly KVX_MAX_CHUNKS records: 128 MiB staged and uploaded) between two device
pools, through kvx_copy_batch with the table's launch and with the staged
kernel forced, compared whole-pool with the oracle; one more chunk is refused
before anything is enqueued.
"""

import numpy as np
import pytest
import torch

import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools

pytestmark = pytest.mark.gpu

N = kvx.KVX_MAX_CHUNKS
SLOT = 8
BODY = N * SLOT  # 32 MiB


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def batch():
    g = np.random.default_rng([W.SEED, 100])
    so = (g.permutation(N) * SLOT).astype(np.uint64)
    do = (g.permutation(N) * SLOT).astype(np.uint64)
    return W.Batch("src", "dst", so, do, np.full(N, SLOT, dtype=np.uint64), "d2d")


@pytest.mark.parametrize("launch", [None, {"variant": "stage"}])
def test_max_chunks_in_one_batch(batch, launch):
    p = Pools({"src": W.PoolSpec("src", "device", BODY, "random", (100,)),
               "dst": W.PoolSpec("dst", "device", BODY, "canary")})
    try:
        want = p.expected([batch])
        s, d, z = p.addrs(batch)
        assert kvx.kvx_plan_chunks(s[:1], d[:1], z[:1]).size == 1  # one chunk per descriptor
        kvx.kvx_copy_batch_ex(s, d, z, None, "d2d", launch, None)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
        # one chunk more than the limit: refused, nothing enqueued
        p.bufs["dst"].fill_(W.CANARY)
        torch.cuda.synchronize()
        before = {name: p.snapshot(name) for name in p.specs}
        s1, d1, z1 = (np.append(a, a[:1]) for a in (s, d, z))
        d1[-1] = np.uint64(p.base("dst") + BODY)  # the trailing guard band: allocated, never written
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_copy_batch_ex(s1, d1, z1, None, "d2d", launch, None)
        assert e.value.status == kvx.KVX_ERR_CAPACITY
        kvx.kvx_stream_check(None)
        p.assert_equal(before)
    finally:
        p.close()

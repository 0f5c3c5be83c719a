"""Host threads calling the C ABI at once, each on its own stream, all bit-exact.

ctypes releases the GIL during each call, so these threads really run
kvx_copy_batch (staging ring, worker pool, status tokens and error flags) concurrently.
"""

import threading

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("threads", [2, 6])
def test_concurrent_callers(threads):
    # one kv_burst pool pair, every thread owning a disjoint set of batches
    w = W.kv_burst(n_sets=2 * threads, n_per_dir=8192, pool_bytes=W.GIB)
    p = Pools(w.pools)
    try:
        batches = [b for pair in w.batches for b in pair]
        want = p.expected(batches)
        errors = []
        per_thread = [batches[i::threads] for i in range(threads)]

        def worker(mine):
            try:
                torch.cuda.set_device(0)
                s = torch.cuda.Stream()
                descs = kvx.Descriptors(8192)
                toks = []
                for k, b in enumerate(mine):
                    if k % 3 == 0:
                        kvx.kvx_copy_batch(*p.addrs(b), None, b.direction, 0, s)
                    elif k % 3 == 1:
                        descs.set(*p.addrs(b)).copy_batch(b.direction, 0, s)
                    else:
                        t = kvx.Transfer()
                        t.start(*p.addrs(b), b.direction, 3000, stream=s)
                        while not t.poll():
                            pass
                        t.close()
                    toks.append(kvx.kvx_status_enqueue(s))
                for t in toks:
                    kvx.kvx_status_wait(t)
            except Exception as e:  # surfaced below
                errors.append(repr(e))

        ts = [threading.Thread(target=worker, args=(m,)) for m in per_thread]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert not errors, errors
        torch.cuda.synchronize()
        p.assert_equal(want)
    finally:
        p.close()


def test_threads_share_one_descriptor_buffer():
    # Four threads copy the same uploaded H2D buffer (units taken from the table's
    # counter) on their own streams. The buffer serialises their calls and orders
    # each copy after the previous one, so no two copies share the counter: after
    # all of them, one more copy into a fresh canary pool must still be exact.
    w = W.kv_burst(n_sets=1, n_per_dir=8192, pool_bytes=W.GIB // 4)
    p = Pools(w.pools)
    try:
        h2d = w.batches[0][0]
        want = p.expected([h2d])
        buf = kvx.DescBuf(h2d.n)
        buf.upload(*p.addrs(h2d), "h2d")
        torch.cuda.synchronize()
        launch = {"variant": "ldg", "assign": "dynamic", "cta_budget": 16}
        errors = []

        def worker():
            try:
                torch.cuda.set_device(0)
                s = torch.cuda.Stream()
                for _ in range(25):
                    buf.copy(stream=s, launch=launch)
                kvx.kvx_stream_check(s)
            except Exception as e:  # surfaced below
                errors.append(repr(e))

        ts = [threading.Thread(target=worker) for _ in range(4)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert not errors, errors
        torch.cuda.synchronize()
        p.assert_equal(want)
        p.bufs["dev"].fill_(W.CANARY)
        torch.cuda.synchronize()
        want = p.expected([h2d])
        buf.copy(launch=launch)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
        buf.close()
    finally:
        p.close()

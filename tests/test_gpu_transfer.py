"""Tail-bounded submission (kvx_transfer): pieces after completion, same bytes as one batch."""

import time

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


def _drive(transfers, limit_s=30.0):
    """Poll every transfer until all report done; return the polls that found work in flight."""
    busy = 0
    t0 = time.perf_counter()
    while True:
        done = [t.poll() for t in transfers]
        if all(done):
            return busy
        busy += 1
        assert time.perf_counter() - t0 < limit_s, "transfer did not finish"
        time.sleep(20e-6)


@pytest.mark.parametrize("chunk", [0, 1000, 2048, 16384])
def test_chunked_bidirectional_burst(chunk):
    w = W.kv_burst(n_sets=1, n_per_dir=16_384, pool_bytes=256 * W.MIB)
    h2d, d2h = w.batches[0]
    p = Pools(w.pools)
    th, td = kvx.Transfer(), kvx.Transfer()
    try:
        want = p.expected([h2d, d2h])
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        th.start(*p.addrs(h2d), "h2d", chunk, stream=s1)
        td.start(*p.addrs(d2h), "d2h", chunk, stream=s2)
        if chunk and chunk < h2d.n:
            assert th.progress() == (chunk, h2d.n)  # only the first piece is out
        _drive([th, td])
        assert th.progress() == (h2d.n, h2d.n) and td.progress() == (d2h.n, d2h.n)
        kvx.kvx_stream_check(s1)
        kvx.kvx_stream_check(s2)
        p.assert_equal(want)
    finally:
        th.close()
        td.close()
        p.close()


def test_transfer_owns_its_descriptors_and_refuses_overlap_in_time():
    w = W.sweep_cell(16, 4096, "d2d")
    (b,) = w.batches
    p = Pools(w.pools)
    t = kvx.Transfer()
    try:
        want = p.expected([b])
        s, d, z = (a.copy() for a in p.addrs(b))
        t.start(s, d, z, "d2d", 512)
        s[:] = 0  # the caller's arrays may be reused at once
        d[:] = 0
        with pytest.raises(kvx.KvxError) as e:  # a second start while a piece is in flight
            t.start(*p.addrs(b), "d2d", 512)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
        _drive([t])
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        t.close()
        p.close()


def test_one_transfer_polled_from_several_threads():
    # Three threads poll the same transfer while the main thread reads its progress:
    # the transfer's lock makes them take turns, so every piece is submitted once,
    # after the previous one completed, and the bytes match the oracle.
    import threading
    w = W.kv_burst(n_sets=1, n_per_dir=16_384, pool_bytes=256 * W.MIB)
    h2d = w.batches[0][0]
    p = Pools(w.pools)
    t = kvx.Transfer()
    try:
        want = p.expected([h2d])
        s = torch.cuda.Stream()
        t.start(*p.addrs(h2d), "h2d", 1000, stream=s)
        errors, seen = [], []

        def poller():
            try:
                t0 = time.perf_counter()
                while not t.poll():
                    assert time.perf_counter() - t0 < 30.0, "transfer did not finish"
            except Exception as e:  # surfaced below
                errors.append(repr(e))

        ts = [threading.Thread(target=poller) for _ in range(3)]
        for th in ts:
            th.start()
        while any(th.is_alive() for th in ts):
            seen.append(t.progress()[0])
        for th in ts:
            th.join()
        assert not errors, errors
        assert t.progress() == (h2d.n, h2d.n)
        assert seen == sorted(seen) and all(x % 1000 == 0 or x == h2d.n for x in seen)
        kvx.kvx_stream_check(s)
        p.assert_equal(want)
    finally:
        t.close()
        p.close()

"""Dynamic work assignment: the LDG kernel's unit counter lives in the chunk table.

Each copy over a table must find the counter zero and leave it zero: the
last warp to finish resets it. So every test here copies over the same table
several times, refilling the destination with the canary in between, so that
a copy that found a stale counter (and skipped units) leaves canary bytes the
oracle does not expect.
"""

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


def _case(direction, n, seed, max_kib=40):
    g = np.random.default_rng([W.SEED, 95, seed])
    slot = (max_kib + 1) * 1024
    sizes = (8 * g.integers(1, max_kib * 128 + 1, n)).astype(np.uint64)
    src = (g.permutation(2 * n)[:n] * slot + 8 * g.integers(0, 2, n)).astype(np.uint64)
    dst = (g.permutation(2 * n)[:n] * slot + 8 * g.integers(0, 2, n)).astype(np.uint64)
    body = 2 * n * slot
    ws = "host" if direction == "h2d" else "device"
    wd = "host" if direction == "d2h" else "device"
    specs = {"src": W.PoolSpec("src", ws, body, "random", (95, seed)),
             "dst": W.PoolSpec("dst", wd, body, "canary")}
    return specs, W.Batch("src", "dst", src, dst, sizes, direction)


def _recanary(p):
    b = p.bufs["dst"]
    if isinstance(b, kvx.HostBuffer):
        b.numpy()[:] = W.CANARY
    else:
        b.fill_(W.CANARY)
    torch.cuda.synchronize()


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("n,budget", [(3, 64), (500, 16), (4000, 64), (4000, 300)])
def test_table_reused_with_dynamic_assignment(direction, n, budget):
    # (3, 64): under 8 units a warp, so assigned by position even when dynamic is asked
    specs, b = _case(direction, n, n + budget)
    p = Pools(specs)
    buf = kvx.DescBuf(max(1, int(sum(-(-int(x) // 16384) for x in b.sizes))))
    try:
        buf.upload(*p.addrs(b), direction)
        for k, assign in enumerate(["dynamic", "dynamic", "static", "dynamic", "dynamic"]):
            _recanary(p)
            want = p.expected([b])
            buf.copy(stream=None, launch={"variant": "ldg", "cta_budget": budget, "assign": assign,
                                          "threads": [128, 256, 512][k % 3]})
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        buf.close()
        p.close()


def test_table_copied_from_two_streams():
    # the second stream's copy waits for the first one's (they share a counter)
    specs, b = _case("h2d", 3000, 7)
    p = Pools(specs)
    buf = kvx.DescBuf(int(sum(-(-int(x) // 16384) for x in b.sizes)))
    try:
        buf.upload(*p.addrs(b), "h2d")
        torch.cuda.synchronize()
        want = p.expected([b])
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        for k in range(6):
            buf.copy(stream=s1 if k % 2 == 0 else s2, launch={"assign": "dynamic", "cta_budget": 32})
        toks = [kvx.kvx_status_enqueue(s) for s in (s1, s2)]
        for t in toks:
            kvx.kvx_status_wait(t)
        torch.cuda.synchronize()
        p.assert_equal(want)
        # and once more after a canary refill: the counter was left zero
        _recanary(p)
        buf.copy(stream=s2, launch={"assign": "dynamic"})
        kvx.kvx_stream_check(s2)
        p.assert_equal(want)
    finally:
        buf.close()
        p.close()


def test_graph_replays_with_dynamic_assignment():
    specs, b = _case("d2h", 2000, 9)
    p = Pools(specs)
    buf = kvx.DescBuf(int(sum(-(-int(x) // 16384) for x in b.sizes)))
    try:
        buf.upload(*p.addrs(b), "d2h")
        torch.cuda.synchronize()
        gs = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            buf.copy(stream=gs, launch={"assign": "dynamic", "cta_budget": 48})
        for _ in range(4):
            _recanary(p)
            want = p.expected([b])
            graph.replay()
            torch.cuda.synchronize()
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        buf.close()
        p.close()


@pytest.mark.parametrize("direction", ["h2d", "d2h"])
def test_ring_and_noalloc_back_to_back(direction):
    # kvx_copy_batch and kvx_copy_batch_noalloc upload a zero header with every
    # table; many calls in a row on one stream, each checked
    specs, b = _case(direction, 1500, 11)
    p = Pools(specs)
    try:
        s = torch.cuda.Stream()
        for k in range(10):
            _recanary(p)
            want = p.expected([b])
            if k % 2:
                kvx.kvx_copy_batch_noalloc(*p.addrs(b), None, direction, 0, s)
            else:
                kvx.kvx_copy_batch_ex(*p.addrs(b), None, direction, {"assign": "dynamic"}, s)
            kvx.kvx_stream_check(s)
            p.assert_equal(want)
    finally:
        p.close()

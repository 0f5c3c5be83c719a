"""Stream order of back-to-back batches whose chunk tables upload on a side stream.

kvx_copy_batch uploads its chunk table on a library side stream when the
caller's stream still has work queued. Each copy must still run after every
earlier copy on the stream: here a chain of batches, submitted without a
synchronisation between them, moves data host -> device -> device -> ... ->
host, each hop reading what the previous hop wrote and the last hops
overwriting pools that earlier hops read. The oracle applies the same hops in
order on host snapshots.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools

pytestmark = pytest.mark.gpu

SLOT = 32 * 1024
N_SLOTS = 2048
BODY = SLOT * N_SLOTS  # 64 MiB per pool


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _hop(g, src, dst, direction, n):
    sizes = (8 * g.integers(1, 3 * 1024 + 1, n)).astype(np.uint64)  # 8 B .. 24 KiB
    s = (g.permutation(N_SLOTS)[:n] * SLOT + 8 * g.integers(0, 2, n)).astype(np.uint64)
    d = (g.permutation(N_SLOTS)[:n] * SLOT + 8 * g.integers(0, 2, n)).astype(np.uint64)
    return W.Batch(src, dst, s, d, sizes, direction)


def _chain(seed):
    g = np.random.default_rng([W.SEED, 91, seed])
    hops = [("h0", "p0", "h2d"), ("p0", "p1", "d2d"), ("p1", "p2", "d2d"), ("p2", "p3", "d2d"),
            ("p3", "p0", "d2d"),   # overwrites the pool the second hop read
            ("p0", "h1", "d2h"), ("h1", "p1", "h2d"), ("p1", "h0", "d2h"),  # h0 was the first source
            ("h0", "p2", "h2d"), ("p2", "p3", "d2d"), ("p3", "h1", "d2h")]
    return [_hop(g, s, d, direction, int(g.choice([300, 1200, 2048]))) for s, d, direction in hops]


@pytest.mark.parametrize("seed", range(3))
def test_chain_on_one_stream(seed):
    specs = {"h0": W.PoolSpec("h0", "host", BODY, "random", (91, seed, 0)),
             "h1": W.PoolSpec("h1", "host", BODY, "canary"),
             "big_s": W.PoolSpec("big_s", "host", 4 * BODY, "random", (91, seed, 1)),
             "big_d": W.PoolSpec("big_d", "device", 4 * BODY, "canary")}
    for k in range(4):
        specs[f"p{k}"] = W.PoolSpec(f"p{k}", "device", BODY, "canary" if k else "random", (91, seed, 2))
    p = Pools(specs)
    try:
        chain = _chain(seed)
        # a long copy first, so that the chain's tables find the stream busy
        big = W.Batch("big_s", "big_d", np.arange(0, 4 * BODY, 1 << 20, dtype=np.uint64),
                      np.arange(0, 4 * BODY, 1 << 20, dtype=np.uint64),
                      np.full(4 * BODY >> 20, 1 << 20, dtype=np.uint64), "h2d")
        want = {name: p.snapshot(name) for name in specs}
        gd = np.uint64(W.GUARD)
        for b in [big] + chain:
            src = want[b.src_pool].copy()
            oracle.copy_batch(want[b.dst_pool], src, b.src_off + gd, b.dst_off + gd, b.sizes)
        s = torch.cuda.Stream()
        toks = []
        for b in [big] + chain:
            kvx.kvx_copy_batch(*p.addrs(b), None, b.direction, 0, s)
            toks.append(kvx.kvx_status_enqueue(s))
        for t in toks:
            kvx.kvx_status_wait(t)
        s.synchronize()
        p.assert_equal(want)
    finally:
        p.close()


def test_descriptors_reused_while_in_flight():
    # One Descriptors object refilled for every call: its arrays are packed
    # before kvx_copy_batch returns, so refilling them at once is safe even
    # while the earlier copies (and their side-stream uploads) are in flight.
    specs = {"h0": W.PoolSpec("h0", "host", BODY, "random", (92,)),
             "p0": W.PoolSpec("p0", "device", BODY, "canary")}
    p = Pools(specs)
    try:
        g = np.random.default_rng([W.SEED, 92])
        slots = g.permutation(N_SLOTS)
        batches = []
        for k in range(16):  # 16 calls: twice round the 8-slot staging ring
            sl = slots[k * 128:(k + 1) * 128]
            off = (sl * SLOT).astype(np.uint64)
            batches.append(W.Batch("h0", "p0", off, off, np.full(128, SLOT, dtype=np.uint64), "h2d"))
        want = p.expected(batches)
        descs = kvx.Descriptors(128)
        s = torch.cuda.Stream()
        for b in batches:
            descs.set(*p.addrs(b)).copy_batch("h2d", 0, s)
        kvx.kvx_stream_check(s)
        p.assert_equal(want)
    finally:
        p.close()

"""Descriptor lists that live on the device: parity with the oracle, graph replay, device-side errors."""

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


class DevArrays:
    """Device copies of a batch's absolute addresses plus its count, at fixed device addresses."""

    def __init__(self, capacity):
        self.src = torch.zeros(capacity, dtype=torch.int64, device="cuda")
        self.dst = torch.zeros(capacity, dtype=torch.int64, device="cuda")
        self.sizes = torch.zeros(capacity, dtype=torch.int64, device="cuda")
        self.count = torch.zeros(1, dtype=torch.int32, device="cuda")

    def fill(self, s, d, z, count=None):
        n = len(z)
        for t, a in ((self.src, s), (self.dst, d), (self.sizes, z)):
            t[:n].copy_(torch.from_numpy(np.asarray(a, dtype=np.uint64).view(np.int64)))
        self.count.fill_(n if count is None else count)

    def ptrs(self):
        return self.src.data_ptr(), self.dst.data_ptr(), self.sizes.data_ptr(), self.count.data_ptr()


def test_moe_calls_from_device_lists():
    m = W.MoeGather(n_slots=400)
    p = Pools(m.pools)
    lst = kvx.DeviceList(192)
    arr = DevArrays(192)
    try:
        for _ in range(3):
            b = m.next_call()
            want = p.expected([b])
            arr.fill(*p.addrs(b))
            lst.copy(*arr.ptrs(), "h2d")
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        lst.close()
        p.close()


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("odd", [False, True])
@pytest.mark.parametrize("assign", ["static", "dynamic"])
def test_sweep_cells_from_device_lists(direction, odd, assign):
    w = W.sweep_cell(24, 1500, direction, odd_tails=odd)
    (b,) = w.batches
    p = Pools(w.pools)
    lst = kvx.DeviceList(8192)
    arr = DevArrays(8192)
    try:
        # twice over the same list: the plan kernel re-zeroes the unit counter
        for _ in range(2):
            dstbuf = p.bufs["dst"]
            if isinstance(dstbuf, kvx.HostBuffer):
                dstbuf.numpy()[:] = W.CANARY
            else:
                dstbuf.fill_(W.CANARY)
            torch.cuda.synchronize()
            want = p.expected([b])
            arr.fill(*p.addrs(b))
            lst.copy(*arr.ptrs(), direction, launch={"cta_budget": 13, "unroll": 4, "assign": assign})
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        lst.close()
        p.close()


def test_large_list_searched_in_global_memory():
    """More than 4,095 descriptors: the chunk scan is searched in global memory."""
    w = W.kv_burst(n_sets=1, n_per_dir=6000, pool_bytes=64 * W.MIB)
    h2d, _ = w.batches[0]
    p = Pools(w.pools)
    lst = kvx.DeviceList(6000)
    arr = DevArrays(6000)
    try:
        want = p.expected([h2d])
        arr.fill(*p.addrs(h2d))
        lst.copy(*arr.ptrs(), "h2d")
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        lst.close()
        p.close()


def test_graph_replay_copies_current_list_contents():
    m = W.MoeGather(n_slots=400)
    p = Pools(m.pools)
    lst = kvx.DeviceList(192)
    arr = DevArrays(192)
    try:
        s = torch.cuda.Stream()
        first = m.next_call()
        arr.fill(*p.addrs(first))
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            lst.copy(*arr.ptrs(), "h2d", stream=s)
        torch.cuda.synchronize()
        assert np.all(p.snapshot("dev") == W.CANARY)  # capture ran nothing
        for k in range(3):
            b = m.next_call()
            if k == 1:  # a shorter list: only the first 5 experts (30 rows)
                b = W.Batch(b.src_pool, b.dst_pool, b.src_off[:30], b.dst_off[:30], b.sizes[:30], "h2d")
            want = p.expected([b])
            arr.fill(*p.addrs(b))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        lst.close()
        p.close()


def test_count_above_capacity_is_clamped_and_reported():
    w = W.sweep_cell(8, 64, "d2d")
    (b,) = w.batches
    p = Pools(w.pools)
    lst = kvx.DeviceList(40)
    arr = DevArrays(64)
    try:
        first40 = W.Batch(b.src_pool, b.dst_pool, b.src_off[:40], b.dst_off[:40], b.sizes[:40], "d2d")
        want = p.expected([first40])
        arr.fill(*p.addrs(b))  # count = 64 > 40
        lst.copy(*arr.ptrs(), "d2d")
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_stream_check(None)
        assert e.value.status == kvx.KVX_ERR_DEVICE_FAULT and "capacity" in str(e.value)
        p.assert_equal(want)
        kvx.kvx_stream_check(None)  # the bit was cleared
    finally:
        lst.close()
        p.close()


def test_bad_descriptor_is_skipped_and_reported():
    w = W.sweep_cell(8, 32, "d2d")
    (b,) = w.batches
    p = Pools(w.pools)
    lst = kvx.DeviceList(32)
    arr = DevArrays(32)
    try:
        sizes = b.sizes.copy()
        sizes[7] = 8188  # not a multiple of 8
        good = np.ones(32, bool)
        good[7] = False
        want = p.expected([W.Batch(b.src_pool, b.dst_pool, b.src_off[good], b.dst_off[good], b.sizes[good], "d2d")])
        s_, d_, _ = p.addrs(b)
        arr.fill(s_, d_, sizes)
        lst.copy(*arr.ptrs(), "d2d")
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_stream_check(None)
        assert e.value.status == kvx.KVX_ERR_DEVICE_FAULT and "validation" in str(e.value)
        p.assert_equal(want)
    finally:
        lst.close()
        p.close()


def test_empty_list_and_host_errors():
    w = W.sweep_cell(8, 16, "d2d")
    p = Pools(w.pools)
    lst = kvx.DeviceList(16)
    arr = DevArrays(16)
    try:
        want = p.expected([])
        arr.fill(*p.addrs(w.batches[0]), count=0)
        lst.copy(*arr.ptrs(), "d2d")
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
        ps, pd, pz, pc = arr.ptrs()
        for bad, status in (((0, pd, pz, pc), kvx.KVX_ERR_INVALID_ARG), ((ps + 4, pd, pz, pc), kvx.KVX_ERR_ALIGN)):
            with pytest.raises(kvx.KvxError) as e:
                lst.copy(*bad, "d2d")
            assert e.value.status == status
        with pytest.raises(kvx.KvxError) as e:
            lst.copy(*arr.ptrs(), "d2d", launch={"variant": "bulk"})
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    finally:
        lst.close()
        p.close()


def test_one_list_copied_from_two_streams():
    # Calls of one list alternate between two streams, each with its own arrays and
    # count: the list's scratch (plan results, chunk offsets) serves one copy at a
    # time, so each call waits for the list's previous copy on the other stream.
    specs = {"src": W.PoolSpec("src", "device", 64 * W.MIB, "random", (99,)),
             "dst": W.PoolSpec("dst", "device", 64 * W.MIB, "canary")}
    p = Pools(specs)
    lst = kvx.DeviceList(4096)
    g = np.random.default_rng([W.SEED, 99])
    slots = g.permutation(4096)  # 16 KiB slots of the destination, split over the calls
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    arrays, batches, used = [], [], 0
    try:
        for k in range(6):
            n = int(g.integers(200, 600))
            so = (g.permutation(4096)[:n] * 16384 + 8 * g.integers(0, 2, n)).astype(np.uint64)
            do = (slots[used:used + n] * 16384 + 8 * g.integers(0, 2, n)).astype(np.uint64)
            used += n
            sz = (8 * g.integers(1, 2047, n)).astype(np.uint64)
            batches.append(W.Batch("src", "dst", so, do, sz, "d2d"))
        want = p.expected(batches)
        for k, b in enumerate(batches):
            a = DevArrays(b.n)
            a.fill(*p.addrs(b))
            arrays.append(a)
        torch.cuda.synchronize()
        for k, a in enumerate(arrays):
            lst.copy(*a.ptrs(), "d2d", stream=streams[k % 2])
        for s in streams:
            kvx.kvx_stream_check(s)
        p.assert_equal(want)
    finally:
        lst.close()
        p.close()


def test_list_of_more_than_4096_tiles():
    # 1,100,000 descriptors: 4,297 plan tiles of 256, more than the copy kernel keeps in
    # shared memory, so the tile bases are searched in global memory
    n = 1_100_000
    specs = {"src": W.PoolSpec("src", "device", 2 * n * 8, "random", (101,)),
             "dst": W.PoolSpec("dst", "device", 2 * n * 8, "canary")}
    p = Pools(specs)
    lst = kvx.DeviceList(n)
    arr = DevArrays(n)
    try:
        g = np.random.default_rng([W.SEED, 101])
        so = (g.permutation(2 * n)[:n] * 8).astype(np.uint64)
        do = (g.permutation(2 * n)[:n] * 8).astype(np.uint64)
        sz = np.full(n, 8, dtype=np.uint64)
        sz[g.random(n) < 0.01] = 0  # zero-size descriptors inside tiles
        b = W.Batch("src", "dst", so, do, sz, "d2d")
        want = p.expected([b])
        arr.fill(*p.addrs(b))
        lst.copy(*arr.ptrs(), "d2d")
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        lst.close()
        p.close()


def test_tiles_without_chunks_are_skipped():
    # whole tiles of zero-size descriptors between tiles that copy: the tile search must land on
    # the tile that holds each chunk, not on an empty one sharing its base
    n = 256 * 12
    specs = {"src": W.PoolSpec("src", "device", 4 * W.MIB, "random", (102,)),
             "dst": W.PoolSpec("dst", "device", 4 * W.MIB, "canary")}
    p = Pools(specs)
    lst = kvx.DeviceList(n)
    arr = DevArrays(n)
    try:
        g = np.random.default_rng([W.SEED, 102])
        so = (g.permutation(4 * W.MIB // 1024)[:n] * 1024).astype(np.uint64)
        do = (g.permutation(4 * W.MIB // 1024)[:n] * 1024).astype(np.uint64)
        sz = (8 * g.integers(1, 129, n)).astype(np.uint64)
        for t in (0, 3, 4, 7, 11):  # empty tiles, the first and the last among them
            sz[t * 256:(t + 1) * 256] = 0
        b = W.Batch("src", "dst", so, do, sz, "d2d")
        want = p.expected([b])
        arr.fill(*p.addrs(b))
        lst.copy(*arr.ptrs(), "d2d")
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        lst.close()
        p.close()

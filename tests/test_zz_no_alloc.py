"""kvx_copy_batch_noalloc gives the same bytes as kvx_copy_batch, two calls in a row.

Who needs it: callers that cannot let a copy allocate memory. A serving engine
that reserves nearly all HBM for its KV cache at start-up makes any later
cudaMalloc fail, and a decode loop with a fixed per-step time budget cannot
absorb an allocation, or the device-wide synchronisation of a cudaFree, in the
middle of a step. kvx_copy_batch allocates its staging ring lazily, so those
callers use kvx_copy_batch_noalloc, whose chunk tables are two fixed 2 MiB
arrays in the library's own device memory, filled in turn.

What is checked: the same two batches (a KV-style 4 KiB batch, then an odd-tail
batch that needs fewer chunks, so the second call runs over a table still
holding the first call's tail) go once through kvx_copy_batch into one
destination pool and once through kvx_copy_batch_noalloc into an identical
pool; the two pools must match byte for byte (the bit-exact tolerance of every
copy test here), and both must match the oracle. A batch one chunk too large
is refused before anything is enqueued, and so is a call during stream capture.
Calls alternating between two busy streams, so that each upload runs on the
side stream while copies on both streams still read the tables, match the
oracle too. At each validation level (0: the fused validate-and-pack pass;
1 and 2: the two-pass path) a valid batch is exact, and a misaligned size or
overlapping destinations are refused with nothing enqueued.

This file sorts last so that a run stopping at its first failure has run every
other test first; it also passes alone in a fresh process.
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


def _batches():
    kv = W.kv_burst(n_sets=1, n_per_dir=4096, pool_bytes=64 * W.MIB)
    first = kv.batches[0][0]                       # 4,096 x 4 KiB, host -> device
    odd = W.sweep_cell(28, 300, "h2d", odd_tails=True).batches[0]   # 300 odd-tail descriptors
    return first, odd


def test_noalloc_matches_copy_batch_two_calls_in_a_row():
    first, odd = _batches()
    body = 64 * W.MIB
    specs = {
        "src": W.PoolSpec("src", "host", body, "random", (77,)),
        "dst_ref": W.PoolSpec("dst_ref", "device", body, "canary"),
        "dst_na": W.PoolSpec("dst_na", "device", body, "canary"),
    }
    p = Pools(specs)
    try:
        def addrs(b, dst):
            return (b.src_off + np.uint64(p.base("src")), b.dst_off + np.uint64(p.base(dst)), b.sizes)

        calls = [W.Batch("src", "dst_na", b.src_off, b.dst_off, b.sizes, "h2d") for b in (first, odd)]
        want = p.expected(calls)["dst_na"]
        stream = torch.cuda.current_stream()
        for b in (first, odd):
            kvx.kvx_copy_batch(*addrs(b, "dst_ref"), None, "h2d", 0, stream)
        for b in (first, odd):                     # two calls in a row on one stream
            kvx.kvx_copy_batch_noalloc(*addrs(b, "dst_na"), None, "h2d", 0, stream)
        kvx.kvx_stream_check(stream)
        ref, got = p.snapshot("dst_ref"), p.snapshot("dst_na")
        assert np.array_equal(got, ref), f"{int(np.count_nonzero(got != ref))} bytes differ from kvx_copy_batch"
        assert np.array_equal(got, want), "differs from the oracle"
    finally:
        p.close()


def test_noalloc_refuses_more_than_its_table():
    p = Pools({"src": W.PoolSpec("src", "device", 4 * W.MIB, "random", (78,)),
               "dst": W.PoolSpec("dst", "device", 4 * W.MIB, "canary")})
    try:
        before = p.snapshot("dst")
        n = kvx.KVX_NOALLOC_MAX_CHUNKS + 1        # 8-byte descriptors: one chunk each
        s = np.full(n, p.base("src"), dtype=np.uint64) + (np.arange(n, dtype=np.uint64) % 1024) * np.uint64(8)
        d = np.uint64(p.base("dst")) + np.arange(n, dtype=np.uint64) * np.uint64(8)
        z = np.full(n, 8, dtype=np.uint64)
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_copy_batch_noalloc(s, d, z, None, "d2d", 0, None)
        assert e.value.status == kvx.KVX_ERR_CAPACITY
        torch.cuda.synchronize()
        assert np.array_equal(p.snapshot("dst"), before)
    finally:
        p.close()


def test_noalloc_refused_inside_capture():
    # The upload reads the one shared host array: a captured upload would read
    # it again at replay time, after other calls had packed other records there.
    p = Pools({"src": W.PoolSpec("src", "device", 4 * W.MIB, "random", (79,)),
               "dst": W.PoolSpec("dst", "device", 4 * W.MIB, "canary")})
    try:
        before = p.snapshot("dst")
        s = np.uint64(p.base("src")) + np.arange(64, dtype=np.uint64) * np.uint64(4096)
        d = np.uint64(p.base("dst")) + np.arange(64, dtype=np.uint64) * np.uint64(4096)
        z = np.full(64, 4096, dtype=np.uint64)
        gs = torch.cuda.Stream()
        x = torch.zeros(16, device="cuda")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            x.add_(1)
            with pytest.raises(kvx.KvxError) as e:
                kvx.kvx_copy_batch_noalloc(s, d, z, None, "d2d", 0, gs)
        assert e.value.status == kvx.KVX_ERR_CAPTURE
        graph.replay()
        torch.cuda.synchronize()
        kvx.kvx_stream_check(None)
        assert float(x[0]) == 1.0                 # the capture itself went on
        assert np.array_equal(p.snapshot("dst"), before)   # and enqueued no copy
    finally:
        p.close()


def test_noalloc_calls_on_two_busy_streams():
    # Twelve H2D batches (disjoint device slots) alternate between two streams.
    # Each stream is kept busy (a 64 MiB device fill queued before every call),
    # so the uploads take the side stream and overlap copies still running on
    # both streams; each upload must wait for the last copy that read its table.
    # A batch copied over another batch's records would leave its own slots at
    # the canary and write the other's twice.
    kv = W.kv_burst(n_sets=12, n_per_dir=2048, pool_bytes=256 * W.MIB)
    batches = [W.Batch("src", "dst", b.src_off, b.dst_off, b.sizes, "h2d") for b, _ in kv.batches]
    body = 256 * W.MIB
    p = Pools({"src": W.PoolSpec("src", "host", body, "random", (80,)),
               "dst": W.PoolSpec("dst", "device", body, "canary")})
    try:
        want = p.expected(batches)
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        filler = [torch.empty(64 * W.MIB, dtype=torch.uint8, device="cuda") for _ in streams]
        torch.cuda.synchronize()
        for i, b in enumerate(batches):
            k = i % 2
            with torch.cuda.stream(streams[k]):
                filler[k].fill_(i)
                kvx.kvx_copy_batch_noalloc(*p.addrs(b), None, "h2d", 0, streams[k])
        torch.cuda.synchronize()
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


@pytest.mark.parametrize("level", [0, 1, 2])
def test_noalloc_validation_levels_and_errors(level):
    # Level 0 takes the fused validate-and-pack pass; levels 1 and 2 the exact
    # two-pass path. Each level copies a valid 4 KiB D2D batch bit-exactly, and
    # refuses, with nothing enqueued, a misaligned size (every level) and
    # overlapping destinations (levels 1 and 2).
    p = Pools({"src": W.PoolSpec("src", "device", 8 * W.MIB, "random", (81,)),
               "dst": W.PoolSpec("dst", "device", 8 * W.MIB, "canary")})
    old = kvx.kvx_get_validate_level()
    try:
        kvx.kvx_set_validate_level(level)
        g = np.random.default_rng([W.SEED, 81, level])
        n = 1024
        so = (g.permutation(2048)[:n] * 4096).astype(np.uint64)
        do = (g.permutation(2048)[:n] * 4096).astype(np.uint64)
        b = W.Batch("src", "dst", so, do, np.full(n, 4096, dtype=np.uint64), "d2d")
        want = p.expected([b])
        kvx.kvx_copy_batch_noalloc(*p.addrs(b), None, "d2d", 0, None)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
        before = {name: p.snapshot(name) for name in p.specs}
        s, d, z = p.addrs(b)
        z_bad = z.copy()
        z_bad[n // 2] = np.uint64(4092)
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_copy_batch_noalloc(s, d, z_bad, None, "d2d", 0, None)
        assert e.value.status == kvx.KVX_ERR_ALIGN
        if level >= 1:
            d_ovl = d.copy()
            d_ovl[n - 1] = d_ovl[0] + np.uint64(8)
            with pytest.raises(kvx.KvxError) as e:
                kvx.kvx_copy_batch_noalloc(s, d_ovl, z, None, "d2d", 0, None)
            assert e.value.status == kvx.KVX_ERR_OVERLAP
        kvx.kvx_stream_check(None)
        p.assert_equal(before)
    finally:
        kvx.kvx_set_validate_level(old)
        p.close()

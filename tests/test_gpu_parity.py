"""GPU parity: every copy through the C ABI is bit-exact against the oracle.

Each test allocates the workload's pools, snapshots them, runs the batch on
the GPU through libkvx.so and compares every byte of every pool (guard bands
and canary included) with the oracle's result on the snapshots.
"""

import numpy as np
import pytest
import torch

import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools, run_batch

pytestmark = pytest.mark.gpu

LDG = {"variant": "ldg"}
BULK = {"variant": "bulk"}
STAGE = {"variant": "stage"}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    kvx.kvx_set_validate_level(1)
    yield
    kvx.kvx_set_validate_level(0)


def _one(pools, batch, **kw):
    want = pools.expected([batch])
    stream = torch.cuda.current_stream()
    run_batch(pools, batch, stream=stream, **kw)
    kvx.kvx_stream_check(stream)
    pools.assert_equal(want)


# ---- config: tiny H2D (1,024 x 4 KiB), full size ---------------------------

@pytest.mark.parametrize("launch", [None, LDG, BULK,
                                    {"variant": "ldg", "cta_budget": 1},
                                    {"variant": "ldg", "cta_budget": 4},
                                    {"variant": "ldg", "cta_budget": 8},
                                    {"variant": "ldg", "cta_budget": 16},
                                    {"variant": "ldg", "cta_budget": 32},
                                    {"variant": "ldg", "cta_budget": 100000},
                                    {"variant": "bulk", "cta_budget": 1},
                                    {"variant": "bulk", "cta_budget": 4},
                                    {"variant": "bulk", "cta_budget": 32, "stages": 2},
                                    {"variant": "bulk", "cta_budget": 8, "stages": 4},
                                    {"variant": "bulk", "cta_budget": 4, "stages": 12},
                                    {"variant": "bulk", "cta_budget": 1, "stages": 7},
                                    STAGE,
                                    {"variant": "stage", "cta_budget": 1, "stages": 2},
                                    {"variant": "stage", "cta_budget": 3, "stages": 8}])
def test_tiny_h2d(launch):
    w = W.tiny_h2d()
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0], launch=launch)
    finally:
        p.close()


@pytest.mark.parametrize("threads", [128, 256, 512])
@pytest.mark.parametrize("unroll", [2, 4, 8])
@pytest.mark.parametrize("policy", [0, 1, 2])
def test_ldg_launch_shapes(threads, unroll, policy):
    w = W.sweep_cell(28, 300, "h2d", odd_tails=True)
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0], launch={"variant": "ldg", "threads": threads, "unroll": unroll,
                                      "store_policy": policy, "cta_budget": 7})
    finally:
        p.close()


# ---- config: KV burst, 16,384 x 4 KiB per direction, H2D || D2H, full size ---

@pytest.mark.parametrize("launch", [None, BULK, STAGE])
def test_kv_burst_bidirectional(launch):
    w = W.kv_burst(n_sets=1)
    p = Pools(w.pools)
    try:
        h2d, d2h = w.batches[0]
        want = p.expected([h2d, d2h])
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        run_batch(p, h2d, stream=s1, launch=launch)
        run_batch(p, d2h, stream=s2, launch=launch)
        kvx.kvx_stream_check(s1)
        kvx.kvx_stream_check(s2)
        p.assert_equal(want)
    finally:
        p.close()


def test_kv_burst_as_bench_times_it():
    """The bench's timed loop, full size: 8 rotating sets of resident tables (kvx_copy_uploaded with the
    table's launch: LDG, units from the counter), the two halves of each burst joined, 12 bursts."""
    import bench
    w = W.kv_burst(n_sets=8)
    p = Pools(w.pools)
    bufs = []
    try:
        batches = [b for pair in w.batches for b in pair]
        want = p.expected(batches)
        s_h, s_d = torch.cuda.Stream(), torch.cuda.Stream()
        for h2d, d2h in w.batches:
            bh, bd = kvx.DescBuf(h2d.n), kvx.DescBuf(d2h.n)
            bh.upload(*p.addrs(h2d), "h2d", s_h)
            bd.upload(*p.addrs(d2h), "d2h", s_d)
            bufs.append((bh, bd))
        assert bufs[0][0].info()[2]["assign"] == kvx.KVX_ASSIGN_DYNAMIC
        join = bench.BurstJoin(torch, s_h, s_d)
        for k in range(12):
            bh, bd = bufs[k % 8]
            bh.copy(stream=s_h)
            bd.copy(stream=s_d)
            join()
        kvx.kvx_stream_check(s_h)
        kvx.kvx_stream_check(s_d)
        p.assert_equal(want)
    finally:
        for bh, bd in bufs:
            bh.close()
            bd.close()
        p.close()


def test_kv_burst_many_sets_ring_reuse():
    """More calls than staging slots, on two streams: every slot is reused."""
    w = W.kv_burst(n_sets=12, n_per_dir=2048, pool_bytes=256 * W.MIB)
    p = Pools(w.pools)
    try:
        want = p.expected([b for pair in w.batches for b in pair])
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        for h2d, d2h in w.batches:
            run_batch(p, h2d, stream=s1)
            run_batch(p, d2h, stream=s2)
        kvx.kvx_stream_check(s1)
        kvx.kvx_stream_check(s2)
        p.assert_equal(want)
    finally:
        p.close()


# ---- config: size / count sweep ----------------------------------------------

@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("odd", [False, True])
@pytest.mark.parametrize("size_kib", W.SWEEP_SIZES_KIB)
@pytest.mark.parametrize("launch", [LDG, BULK, STAGE])
def test_sweep_cells(direction, odd, size_kib, launch):
    w = W.sweep_cell(size_kib, 256, direction, odd_tails=odd)
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0], launch=launch)
    finally:
        p.close()


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("n", [16, 4096, 65536])
def test_sweep_counts_default_launch(direction, n):
    w = W.sweep_cell(4, n, direction, odd_tails=False)
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0])
    finally:
        p.close()


@pytest.mark.parametrize("direction", ["h2d", "d2d"])
def test_sweep_full_size_cell(direction):
    """The largest sweep cell: 8,192 x 64 KiB = 512 MiB."""
    w = W.sweep_cell(64, 65_536, direction, odd_tails=False)
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0])
    finally:
        p.close()


# ---- config: MoE expert-miss gather, full size -----------------------------------

@pytest.mark.parametrize("launch", [None, LDG, BULK, STAGE])
def test_moe_gather(launch):
    m = W.MoeGather()
    p = Pools(m.pools)
    try:
        calls = [m.next_call() for _ in range(3)]
        want = p.expected(calls)
        stream = torch.cuda.current_stream()
        for b in calls:
            run_batch(p, b, stream=stream, launch=launch)
        kvx.kvx_stream_check(stream)
        p.assert_equal(want)
    finally:
        p.close()


# ---- edge cases -------------------------------------------------------------------

def _pools_small(where_src="host", where_dst="device", body=1 << 20):
    return Pools({"src": W.PoolSpec("src", where_src, body, "random", (90,)),
                  "dst": W.PoolSpec("dst", where_dst, body, "canary")})


def _batch(so, do, sz, direction):
    u = lambda a: np.asarray(a, dtype=np.uint64)
    return W.Batch("src", "dst", u(so), u(do), u(sz), direction)


@pytest.mark.parametrize("launch", [LDG, BULK, STAGE])
@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
def test_phase_combinations(direction, launch):
    """Sizes 8..40 and around the chunk size at every (src mod 16, dst mod 16) pair."""
    ws = "host" if direction == "h2d" else "device"
    wd = "host" if direction == "d2h" else "device"
    p = _pools_small(ws, wd, body=2 * W.MIB)
    so, do, sz = [], [], []
    slot = 40 * 1024
    k = 0
    for size in (8, 16, 24, 32, 40, 16376, 16384, 16392, 32768 + 8):
        for sp in (0, 8):
            for dp in (0, 8):
                so.append(k * slot + sp)
                do.append(k * slot + dp)
                sz.append(size)
                k += 1
    try:
        _one(p, _batch(so, do, sz, direction), launch=launch)
    finally:
        p.close()


def test_empty_and_zero_size_batches():
    p = _pools_small()
    try:
        want = p.expected([])
        kvx.kvx_copy_batch([], [], [], None, "h2d", 0, None)
        base = p.base("src")
        kvx.kvx_copy_batch([base, 0], [p.base("dst"), 0], [0, 0], None, "h2d", 0, None)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


@pytest.mark.parametrize("launch", [LDG, BULK, STAGE])
def test_single_large_descriptor(launch):
    """One 64 MiB descriptor (4,096 chunks) and one 8-byte descriptor."""
    p = _pools_small("device", "device", body=80 * W.MIB)
    try:
        _one(p, _batch([0, 70 * W.MIB], [8 * W.MIB, 75 * W.MIB], [64 * W.MIB, 8], "d2d"), launch=launch)
    finally:
        p.close()


def test_same_pool_d2d():
    p = Pools({"pool": W.PoolSpec("pool", "device", 4 * W.MIB, "random", (91,))})
    try:
        b = W.Batch("pool", "pool", np.arange(0, 64, dtype=np.uint64) * 16384,
                    np.arange(64, 128, dtype=np.uint64) * 16384 + 8, np.full(64, 16376, np.uint64), "d2d")
        _one(p, b)
    finally:
        p.close()


# ---- descriptor buffers, graph capture ---------------------------------------------

@pytest.mark.parametrize("variant", ["ldg", "bulk", "stage"])
def test_desc_buf_upload_and_replay(variant):
    w = W.kv_burst(n_sets=2, n_per_dir=4096, pool_bytes=128 * W.MIB)
    p = Pools(w.pools)
    buf = kvx.DescBuf(8192)
    try:
        stream = torch.cuda.current_stream()
        h2d_a, _ = w.batches[0]
        h2d_b, _ = w.batches[1]
        want = p.expected([h2d_a])
        buf.upload(*p.addrs(h2d_a), "h2d", stream)
        n, payload, sel = buf.info()
        assert n == 4096 and payload == 4096 * 4096
        buf.copy(stream=stream, launch={"variant": variant})
        buf.copy(stream=stream, launch={"variant": variant, "cta_budget": 3})  # idempotent replay
        kvx.kvx_stream_check(stream)
        p.assert_equal(want)
        want = p.expected([h2d_b])
        buf.upload(*p.addrs(h2d_b), "h2d", stream)
        buf.copy(stream=stream, launch={"variant": variant})
        kvx.kvx_stream_check(stream)
        p.assert_equal(want)
    finally:
        buf.close()
        p.close()


def test_desc_buf_capacity():
    buf = kvx.DescBuf(4)
    try:
        with pytest.raises(kvx.KvxError) as e:
            buf.upload([1 << 20], [1 << 30], [5 * 16384], "d2d")
        assert e.value.status == kvx.KVX_ERR_CAPACITY
    finally:
        buf.close()


def test_graph_capture_of_uploaded_copy():
    w = W.tiny_h2d()
    p = Pools(w.pools)
    buf = kvx.DescBuf(1024)
    try:
        (b,) = w.batches
        want = p.expected([b])
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            buf.upload(*p.addrs(b), "h2d", s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            buf.copy(stream=s)
            with pytest.raises(kvx.KvxError) as e:  # the host-staging path refuses capture
                run_batch(p, b, stream=s)
            assert e.value.status == kvx.KVX_ERR_CAPTURE
        # capture itself ran nothing: the destination is still all canary
        torch.cuda.synchronize()
        assert np.all(p.snapshot("dev") == W.CANARY)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        buf.close()
        p.close()


# ---- validation with real pointers, baselines, bounded wait ---------------------

def test_validate_level2_address_kinds():
    p = _pools_small()
    try:
        hs, dd = p.base("src"), p.base("dst")
        assert kvx.kvx_validate([hs], [dd], [4096], None, "h2d", 2) == kvx.KVX_OK
        assert kvx.kvx_validate([dd], [hs], [4096], None, "h2d", 2) == kvx.KVX_ERR_NOT_MAPPED
        assert kvx.kvx_validate([hs], [dd], [4096], None, "d2d", 2) == kvx.KVX_ERR_NOT_MAPPED
        assert kvx.kvx_validate([dd], [hs], [4096], None, "d2h", 2) == kvx.KVX_OK
    finally:
        p.close()


def test_overlap_rejected_and_nothing_enqueued():
    p = _pools_small()
    try:
        want = p.expected([])
        hs, dd = p.base("src"), p.base("dst")
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_copy_batch([hs, hs + 8192], [dd, dd + 4088], [4096, 4096], None, "h2d", 0, None)
        assert e.value.status == kvx.KVX_ERR_OVERLAP
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
def test_memcpy_baseline_parity(direction):
    w = W.sweep_cell(8, 256, direction, odd_tails=True)
    p = Pools(w.pools)
    try:
        (b,) = w.batches
        want = p.expected([b])
        s, d, z = p.addrs(b)
        nr = kvx.kvx_copy_batch_memcpy(s, d, z, None, direction, None)
        assert nr == b.n  # shuffled slots: nothing to coalesce
        torch.cuda.synchronize()
        p.assert_equal(want)
    finally:
        p.close()


def test_memcpy_baseline_coalesces_adjacent():
    p = _pools_small()
    try:
        so = np.arange(16, dtype=np.uint64) * 4096
        b = _batch(so, so + np.uint64(65536), np.full(16, 4096), "h2d")
        want = p.expected([b])
        s, d, z = p.addrs(b)
        assert kvx.kvx_copy_batch_memcpy(s, d, z, None, "h2d", None) == 1
        torch.cuda.synchronize()
        p.assert_equal(want)
    finally:
        p.close()


def test_bounded_wait_times_out_and_context_survives():
    stream = torch.cuda.current_stream()
    kvx.kvx_stream_check(stream)  # clear
    kvx.kvx_selftest_wait_timeout(50_000_000, stream)  # 50 ms
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_stream_check(stream)
    assert e.value.status == kvx.KVX_ERR_TIMEOUT
    kvx.kvx_stream_check(stream)  # the bit was cleared
    # the context is still usable
    w = W.tiny_h2d()
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0])
    finally:
        p.close()


# ---- the fused validate+pack path of kvx_copy_batch (validation level 0) ---------

@pytest.fixture
def level0():
    kvx.kvx_set_validate_level(0)
    yield
    kvx.kvx_set_validate_level(1)


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("odd", [False, True])
def test_level0_sweep_cells(level0, direction, odd):
    w = W.sweep_cell(24, 2000, direction, odd_tails=odd)
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0])
    finally:
        p.close()


def test_level0_kv_burst_and_moe(level0):
    w = W.kv_burst(n_sets=2, n_per_dir=8192, pool_bytes=256 * W.MIB)
    p = Pools(w.pools)
    try:
        want = p.expected([b for pair in w.batches for b in pair])
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        for h2d, d2h in w.batches:
            run_batch(p, h2d, stream=s1)
            run_batch(p, d2h, stream=s2)
        kvx.kvx_stream_check(s1)
        kvx.kvx_stream_check(s2)
        p.assert_equal(want)
    finally:
        p.close()
    m = W.MoeGather(n_slots=200)
    p = Pools(m.pools)
    try:
        calls = [m.next_call() for _ in range(2)]
        want = p.expected(calls)
        for b in calls:
            run_batch(p, b)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


def test_level0_batch_larger_than_a_staging_slot(level0):
    """70,000 one-chunk descriptors: more than a fresh slot holds, so the exact path grows it."""
    n = 70_000
    p = _pools_small("device", "device", body=2 * W.MIB)
    try:
        g = np.random.default_rng(5)
        dst = g.permutation(2 * W.MIB // 16)[:n].astype(np.uint64) * np.uint64(16)
        src = g.integers(0, 2 * W.MIB // 8, n).astype(np.uint64) * np.uint64(8)
        _one(p, _batch(src, dst, np.full(n, 8), "d2d"))
    finally:
        p.close()


def test_level0_errors_still_reported(level0):
    p = _pools_small()
    try:
        want = p.expected([])
        hs, dd = p.base("src"), p.base("dst")
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_copy_batch([hs, hs + 8192], [dd, dd + 8192], [4096, 4100], None, "h2d", 0, None)
        assert e.value.status == kvx.KVX_ERR_ALIGN
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_copy_batch([hs, 0], [dd, dd + 8192], [4096, 4096], None, "h2d", 0, None)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


def test_descriptors_helper_parity(level0):
    w = W.kv_burst(n_sets=3, n_per_dir=4096, pool_bytes=128 * W.MIB)
    p = Pools(w.pools)
    try:
        want = p.expected([b for pair in w.batches for b in pair])
        dh, dd = kvx.Descriptors(4096), kvx.Descriptors(4096)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        for h2d, d2h in w.batches:  # refilled in place as soon as each call returns
            dh.set(*p.addrs(h2d)).copy_batch("h2d", 0, s1)
            dd.set(*p.addrs(d2h)).copy_batch("d2h", 0, s2)
        kvx.kvx_stream_check(s1)
        kvx.kvx_stream_check(s2)
        p.assert_equal(want)
    finally:
        p.close()


@pytest.mark.parametrize("policy", ["throughput", "tail"])
@pytest.mark.parametrize("shape", ["few_large", "fragmented", "d2d_odd_large"])
def test_auto_policy_paths(policy, shape):
    direction = "h2d"
    if shape == "d2d_odd_large":  # ~176 MiB of D2D chunks whose phases differ: the table's STAGE kernel
        w = W.sweep_cell(16, 12000, "d2d", odd_tails=True)
        p = Pools(w.pools)
        b = w.batches[0]
        direction = "d2d"
        expect = "kernel_stage" if policy == "throughput" else "kernel_bulk"
    elif shape == "few_large":
        p = _pools_small("host", "device", body=40 * W.MIB)
        b = _batch([0, 12 * W.MIB, 30 * W.MIB], [8 * W.MIB, 20 * W.MIB, 2 * W.MIB], [4 * W.MIB, 3 * W.MIB, W.MIB],
                   "h2d")
        expect = "dma"
    else:
        w = W.sweep_cell(8, 3000, "h2d", odd_tails=True)
        p = Pools(w.pools)
        b = w.batches[0]
        expect = "kernel_ldg" if policy == "throughput" else "kernel_bulk"
    try:
        want = p.expected([b])
        path = kvx.kvx_copy_batch_auto(*p.addrs(b), None, direction, policy, None)
        assert path == expect
        torch.cuda.synchronize()
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


@pytest.mark.parametrize("stages", [2, 5, 12])
@pytest.mark.parametrize("size_kib", [4, 12, 64])
def test_bulk_ring_sizes_with_mixed_alignment(stages, size_kib):
    """Rings cut into stages of the longest chunk; odd-tail chunks mixed in go through the warp path."""
    w = W.sweep_cell(size_kib, 700, "h2d", odd_tails=True)
    (b,) = w.batches
    b.sizes[::3] = size_kib * W.KIB  # a third of the descriptors 16-byte clean again (where aligned)
    p = Pools(w.pools)
    try:
        _one(p, b, launch={"variant": "bulk", "cta_budget": 5, "stages": stages})
    finally:
        p.close()


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("stages", [2, 4, 8])
@pytest.mark.parametrize("budget,policy", [(1, 0), (5, 1), (1216, 2)])
def test_stage_launch_shapes(direction, stages, budget, policy):
    """The STAGE kernel at every ring depth, a few grids and every store policy, on odd-tail chunks of up to
    28 KiB (two chunks each: 16 KiB + the rest, seven 4 KiB units), every phase pair."""
    w = W.sweep_cell(28, 300, direction, odd_tails=True)
    p = Pools(w.pools)
    try:
        _one(p, w.batches[0], launch={"variant": "stage", "stages": stages, "cta_budget": budget,
                                      "store_policy": policy})
    finally:
        p.close()


def test_status_tokens_pipelined():
    """Submit, enqueue a status read, submit more, then collect: the enqueue-only pattern."""
    w = W.kv_burst(n_sets=4, n_per_dir=2048, pool_bytes=64 * W.MIB)
    p = Pools(w.pools)
    try:
        want = p.expected([b for pair in w.batches for b in pair])
        s1 = torch.cuda.Stream()
        toks = []
        for h2d, d2h in w.batches:
            run_batch(p, h2d, stream=s1)
            run_batch(p, d2h, stream=s1)
            toks.append(kvx.kvx_status_enqueue(s1))
        for t in toks:
            kvx.kvx_status_wait(t)
            assert kvx.kvx_status_query(t) is True
        p.assert_equal(want)
    finally:
        p.close()


def test_status_token_refused_inside_capture():
    # a status read waits on the host, so it cannot be part of a graph
    gs = torch.cuda.Stream()
    x = torch.zeros(16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        x.add_(1)
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_status_enqueue(gs)
    assert e.value.status == kvx.KVX_ERR_CAPTURE
    graph.replay()
    kvx.kvx_stream_check(None)
    assert float(x[0]) == 1.0  # the capture itself went on


def test_status_token_pending_then_timeout_then_expiry():
    s = torch.cuda.Stream()
    kvx.kvx_stream_check(s)
    kvx.kvx_selftest_wait_timeout(200_000_000, s)  # 200 ms of GPU work that ends in a timeout bit
    tok = kvx.kvx_status_enqueue(s)
    assert kvx.kvx_status_query(tok) is False  # the stream has not reached the read yet
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_status_wait(tok)
    assert e.value.status == kvx.KVX_ERR_TIMEOUT
    old = kvx.kvx_status_enqueue(s)
    kvx.kvx_status_wait(old)
    for _ in range(1024):
        kvx.kvx_status_enqueue(s)
    torch.cuda.synchronize()
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_status_wait(old)
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG


@pytest.mark.parametrize("n,odd,variant", [(4096, False, "ldg"), (32768, False, "ldg"), (32768, True, "stage"),
                                           (4096, True, "ldg")])
def test_d2d_table_row_follows_shape(n, odd, variant):
    # 16 KiB D2D chunks take LDG when their phases agree (3,648 CTAs at 64 MiB,
    # 9,728 at 512 MiB); with 8-byte phases that differ, a batch of 128 MiB or
    # more takes the STAGE row (480 MiB here) and a smaller one LDG (60 MiB).
    w = W.sweep_cell(16, n, "d2d", odd_tails=odd)
    (b,) = w.batches
    p = Pools(w.pools)
    buf = kvx.DescBuf(int(sum(-(-int(x) // 16384) for x in b.sizes)))
    try:
        buf.upload(*p.addrs(b), "d2d")
        assert buf.info()[2]["variant"] == kvx.VARIANTS[variant]
        want = p.expected([b])
        buf.copy(stream=None)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        buf.close()
        p.close()


def test_nvtx_ranges_on():
    """KVX_NVTX=1 (NVTX ranges around the entry points, no tool attached): the copy is unchanged."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import __graft_entry__ as g\n"
            "g.smoke()\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=root,
                         env=dict(os.environ, KVX_NVTX="1"))
    assert out.returncode == 0 and "smoke ok" in out.stdout, out.stdout + out.stderr

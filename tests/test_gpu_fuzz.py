"""Randomised batches against the oracle: shapes, phases, directions, variants and launch shapes.

Each case draws (from its seed) a descriptor count, sizes that are multiples
of 8 from 8 bytes to 100 KiB (a quarter of them one-chunk 4 KiB pages, some
zero), independent 0/8 start phases, disjoint destinations, possibly
overlapping sources, and a launch configuration (variant, grid, threads,
loads in flight, store policy, work assignment); the whole destination pool
must equal the oracle's.
"""

import numpy as np
import pytest
import torch

import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools, run_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _random_case(seed, matched=False):
    g = np.random.default_rng([W.SEED, 77 if not matched else 78, seed])
    direction = ["h2d", "d2h", "d2d"][seed % 3]
    n = int(g.choice([1, 3, 17, 200, 1500, 5000]))
    kind = g.integers(0, 4, n)
    sizes = np.where(kind == 0, 4096, 8 * g.integers(1, 100 * 1024 // 8 + 1, n)).astype(np.uint64)
    sizes[g.random(n) < 0.03] = 0
    slot = 104 * 1024
    n_slots = 2 * n + 4
    dst_phase = 8 * g.integers(0, 2, n)
    # matched: every descriptor's src and dst agree mod 16 (the phase-matched kernel instance)
    src_phase = dst_phase if matched else 8 * g.integers(0, 2, n)
    dst = (g.permutation(n_slots)[:n] * slot + dst_phase).astype(np.uint64)
    src = (g.integers(0, n_slots, n) * slot + src_phase).astype(np.uint64)  # may repeat
    body = n_slots * slot
    launch = {"variant": str(g.choice(["ldg", "bulk", "stage"])), "cta_budget": int(g.choice([1, 3, 16, 64, 300]))}
    if launch["variant"] == "ldg":
        launch.update(threads=int(g.choice([128, 256, 512])), unroll=int(g.choice([2, 4, 8])),
                      store_policy=int(g.integers(0, 3)), assign=int(g.integers(0, 3)))
    elif launch["variant"] == "bulk":
        launch["stages"] = int(g.integers(2, 13))
    else:
        launch.update(stages=int(g.choice([2, 4, 8])), store_policy=int(g.integers(0, 3)))
    ws = "host" if direction == "h2d" else "device"
    wd = "host" if direction == "d2h" else "device"
    specs = {"src": W.PoolSpec("src", ws, body, "random", (77, seed)),
             "dst": W.PoolSpec("dst", wd, body, "canary")}
    return specs, W.Batch("src", "dst", src, dst, sizes, direction), launch


@pytest.mark.parametrize("seed", range(36))
def test_random_batches(seed):
    specs, b, launch = _random_case(seed)
    p = Pools(specs)
    try:
        want = p.expected([b])
        run_batch(p, b, launch=launch)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


@pytest.mark.parametrize("seed", range(12))
def test_random_phase_matched_batches(seed):
    # heads and tails of 8 bytes, but src and dst in phase: the kernel without re-pairing
    specs, b, launch = _random_case(seed, matched=True)
    p = Pools(specs)
    try:
        want = p.expected([b])
        run_batch(p, b, launch=launch)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


@pytest.mark.parametrize("seed", range(36, 42))
def test_random_batches_noalloc_and_devlist(seed):
    specs, b, _ = _random_case(seed)
    p = Pools(specs)
    try:
        want = p.expected([b])
        s, d, z = p.addrs(b)
        if seed % 2:
            kvx.kvx_copy_batch_noalloc(s, d, z, None, b.direction, 0, None)
        else:
            lst = kvx.DeviceList(max(1, b.n))
            arrs = [torch.from_numpy(a.view(np.int64)).cuda() for a in (s, d, z)]
            cnt = torch.full((1,), b.n, dtype=torch.int32, device="cuda")
            lst.copy(*(t.data_ptr() for t in arrs), cnt.data_ptr(), b.direction)
            torch.cuda.synchronize()
            lst.close()
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()

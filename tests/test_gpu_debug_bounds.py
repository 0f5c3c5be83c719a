"""The kernel-side debug bounds check (kvx_debug_bounds).

With the pools' bodies registered, every copy kernel must skip a chunk whose
source or destination leaves them, report it (KVX_ERR_DEVICE_FAULT), and
copy every other chunk exactly. The stray descriptor here crosses the end of
its pool's body into the pool's guard band: memory that is allocated, so
nothing can fault even if a check failed, and that the oracle expects to stay
canary-filled while the check is on. Every test turns the check off again.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools

pytestmark = pytest.mark.gpu

BODY = 16 * W.MIB
SLOT = 16 * W.KIB  # holds a descriptor of up to 16,376 bytes shifted by 8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)


@pytest.fixture
def bounds_off():
    yield
    kvx.kvx_debug_bounds([], [])


def _setup(direction, seed):
    ws = "host" if direction == "h2d" else "device"
    wd = "host" if direction == "d2h" else "device"
    p = Pools({"src": W.PoolSpec("src", ws, BODY, "random", (96, seed)),
               "dst": W.PoolSpec("dst", wd, BODY, "canary")})
    g = np.random.default_rng([W.SEED, 96, seed])
    n = 600
    size = int(g.choice([4096, 12288, 16376]))
    odd = size % 16 == 8
    so = (g.permutation(BODY // SLOT - 1)[:n] * SLOT + (8 * g.integers(0, 2, n) if odd else 0)).astype(np.uint64)
    do = (g.permutation(BODY // SLOT - 1)[:n] * SLOT).astype(np.uint64)
    sz = np.full(n, size, dtype=np.uint64)
    return p, so, do, sz


def _register(p):
    lo = [p.base("src"), p.base("dst")]
    hi = [p.base("src") + BODY, p.base("dst") + BODY]
    kvx.kvx_debug_bounds(lo, hi)


def _expected(p, so, do, sz, skip):
    want = {name: p.snapshot(name) for name in p.specs}
    keep = np.ones(sz.size, dtype=bool)
    keep[skip] = False
    g = np.uint64(W.GUARD)
    src = want["src"].copy()
    oracle.copy_batch(want["dst"], src, so[keep] + g, do[keep] + g, sz[keep])
    return want


def _stray(which, so, do, sz):
    """Move descriptor 7's source or destination so that it ends 2 KiB past its pool's body: inside the
    guard band (allocated memory), in the last slot, which no other descriptor uses."""
    off = np.uint64(BODY + 2048) - sz[7]
    if which == "dst":
        do[7] = off
    else:
        so[7] = off
    assert 2048 <= W.GUARD
    return 7


@pytest.mark.parametrize("direction,launch", [
    ("d2d", {"variant": "ldg"}),
    ("h2d", {"variant": "ldg", "assign": "dynamic", "cta_budget": 2, "threads": 128}),
    ("d2h", {"variant": "ldg"}),
    ("d2d", {"variant": "bulk", "cta_budget": 16}),
    ("h2d", {"variant": "bulk", "cta_budget": 4}),
    ("d2d", {"variant": "stage"}),
    ("d2h", {"variant": "stage", "stages": 2}),
])
@pytest.mark.parametrize("which", ["dst", "src"])
def test_stray_chunk_is_skipped_and_reported(bounds_off, direction, launch, which):
    p, so, do, sz = _setup(direction, 1 if which == "dst" else 2)
    try:
        _register(p)
        # inside the bounds: copied exactly, no report
        want = _expected(p, so, do, sz, [])
        s, d, z = so + np.uint64(p.base("src")), do + np.uint64(p.base("dst")), sz
        kvx.kvx_copy_batch_ex(s, d, z, None, direction, launch, None)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
        # one descriptor leaves its pool: that chunk is skipped, the rest copied
        bad = _stray(which, so, do, sz)
        want = _expected(p, so, do, sz, [bad])
        s, d = so + np.uint64(p.base("src")), do + np.uint64(p.base("dst"))
        kvx.kvx_copy_batch_ex(s, d, z, None, direction, launch, None)
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_stream_check(None)
        assert e.value.status == kvx.KVX_ERR_DEVICE_FAULT and "debug bounds" in str(e.value)
        p.assert_equal(want)
        assert np.all(p.snapshot("dst")[-W.GUARD:] == W.CANARY)
        # check off: the same batch writes the stray chunk too (into the guard band)
        kvx.kvx_debug_bounds([], [])
        want = _expected(p, so, do, sz, [])
        kvx.kvx_copy_batch_ex(s, d, z, None, direction, launch, None)
        kvx.kvx_stream_check(None)
        p.assert_equal(want)
    finally:
        p.close()


def test_device_list_descriptor_outside_is_skipped(bounds_off):
    p, so, do, sz = _setup("d2d", 3)
    try:
        _register(p)
        bad = _stray("dst", so, do, sz)
        want = _expected(p, so, do, sz, [bad])
        s, d = so + np.uint64(p.base("src")), do + np.uint64(p.base("dst"))
        arrs = [torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).cuda() for a in (s, d, sz)]
        cnt = torch.full((1,), sz.size, dtype=torch.int32, device="cuda")
        lst = kvx.DeviceList(sz.size)
        try:
            lst.copy(arrs[0].data_ptr(), arrs[1].data_ptr(), arrs[2].data_ptr(), cnt.data_ptr(), "d2d")
            with pytest.raises(kvx.KvxError) as e:
                kvx.kvx_stream_check(None)
            assert e.value.status == kvx.KVX_ERR_DEVICE_FAULT and "debug bounds" in str(e.value)
            p.assert_equal(want)
        finally:
            lst.close()
    finally:
        p.close()


def test_bounds_argument_errors(bounds_off):
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_debug_bounds([1 << 20], [1 << 20])
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_debug_bounds(np.arange(65) << 20, (np.arange(65) + 1) << 20)
    assert e.value.status == kvx.KVX_ERR_CAPACITY
    kvx.kvx_debug_bounds(np.arange(64) << 20, (np.arange(64) + 1) << 20)  # the maximum is accepted

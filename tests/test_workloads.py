"""The seeded workloads against the pages' printed figures and their own stated structure (CPU only)."""

import numpy as np
import pytest

import oracle
import workloads as W


def test_moe_banks_closed_form(golden):
    g = golden("moe_banks.txt")
    rows = tuple(int(x) for x in g["row_bytes"])
    assert rows == W.MOE_ROW_BYTES
    assert sum(rows) == int(g["expert_bytes"][0]) == 1_781_760
    assert W.MOE_EXPERTS == int(g["experts"][0])
    assert W.MOE_SLOTS == int(g["slots"][0])
    # bytes-in-flight arithmetic printed on the same page
    assert 6 * 8 * 1024 * 16 == int(g["inflight_ldg_bytes"][0])
    assert 8 * 3 * 16 * 1024 == int(g["inflight_tma_bytes"][0])
    assert 3 * 16 * 1024 == int(g["smem_per_cta_bytes"][0])
    assert 4 * 4 * 16 * 1024 == int(g["inflight_best_bytes"][0])


def test_kv_burst_closed_form(golden):
    g = golden("kv_burst.txt")
    n, b = int(g["descriptors_per_direction"][0]), int(g["descriptor_bytes"][0])
    assert n * b == int(g["bytes_per_direction"][0]) == 64 * W.MIB
    # (64 + 64) MiB per 50 ms period = 2.5 GiB/s
    rate = 2 * n * b / (int(g["burst_period_ms"][0]) / 1000) / W.GIB
    assert rate == pytest.approx(float(g["target_rate_gib_s"][0]))


def test_tiny_h2d_shape():
    w = W.tiny_h2d()
    (b,) = w.batches
    assert b.n == 1024 and b.payload_bytes == 4 * W.MIB
    assert len(set(b.src_off.tolist())) == 1024 and len(set(b.dst_off.tolist())) == 1024
    assert int(b.src_off.max()) + 4096 <= w.pools["host"].body_bytes
    assert int(b.dst_off.max()) + 4096 <= w.pools["dev"].body_bytes
    assert w.pools["dev"].fill == "canary"
    assert oracle.ranges_disjoint(b.dst_off, b.sizes)


def test_kv_burst_sets_disjoint():
    w = W.kv_burst(n_sets=3, n_per_dir=2048, pool_bytes=64 * W.MIB)
    host_ranges, dev_ranges = [], []
    for h2d, d2h in w.batches:
        assert h2d.n == d2h.n == 2048
        host_ranges += [h2d.src_off, d2h.dst_off]
        dev_ranges += [h2d.dst_off, d2h.src_off]
    for ranges in (host_ranges, dev_ranges):
        off = np.concatenate(ranges)
        assert oracle.ranges_disjoint(off, np.full(off.size, 4096, dtype=np.uint64))


def test_kv_burst_is_seeded():
    a = W.kv_burst(n_sets=1, n_per_dir=64, pool_bytes=W.MIB)
    b = W.kv_burst(n_sets=1, n_per_dir=64, pool_bytes=W.MIB)
    assert np.array_equal(a.batches[0][0].src_off, b.batches[0][0].src_off)


@pytest.mark.parametrize("odd", [False, True])
@pytest.mark.parametrize("size_kib", W.SWEEP_SIZES_KIB)
def test_sweep_cell_structure(size_kib, odd):
    w = W.sweep_cell(size_kib, 65_536, "d2d", odd_tails=odd)
    (b,) = w.batches
    assert b.n * size_kib * W.KIB <= W.SWEEP_CAP_BYTES
    assert np.all(b.sizes % 8 == 0) and np.all(b.src_off % 8 == 0) and np.all(b.dst_off % 8 == 0)
    if odd:
        assert np.all(b.sizes % 16 == 8)
        assert np.all(b.sizes <= size_kib * W.KIB - 8)
        assert np.any(b.src_off % 16 == 8) and np.any(b.dst_off % 16 == 0)
    assert int((b.src_off + b.sizes).max()) <= w.pools["src"].body_bytes
    assert int((b.dst_off + b.sizes).max()) <= w.pools["dst"].body_bytes
    assert oracle.ranges_disjoint(b.dst_off, b.sizes)


def test_moe_calls():
    m = W.MoeGather()
    assert m.expert_bytes == 1_781_760
    used = set()
    for _ in range(5):
        b = m.next_call()
        assert b.n == 32 * 6 and b.payload_bytes == 32 * 1_781_760
        assert oracle.ranges_disjoint(b.dst_off, b.sizes)
        assert int((b.src_off + b.sizes).max()) <= m.pools["host"].body_bytes
        assert int((b.dst_off + b.sizes).max()) <= m.pools["dev"].body_bytes
        slots = set(((b.dst_off[::6] - m.cache_base[0]) // W.MOE_ROW_BYTES[0]).tolist())
        assert len(slots) == 32 and not (slots & used)
        used |= slots


def test_fill_pool_seeded_and_canary():
    spec = W.PoolSpec("p", "host", 8192, "random", (9,))
    a = np.zeros(spec.total_bytes, dtype=np.uint8)
    b = np.zeros(spec.total_bytes, dtype=np.uint8)
    W.fill_pool(a, spec)
    W.fill_pool(b, spec)
    assert np.array_equal(a, b) and a.std() > 50
    c = W.PoolSpec("c", "device", 8192, "canary")
    buf = np.zeros(c.total_bytes, dtype=np.uint8)
    W.fill_pool(buf, c)
    assert np.all(buf == 0xA5)

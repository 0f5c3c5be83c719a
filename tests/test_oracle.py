"""Pins of the oracle to things other than itself (CPU only).

* A per-byte brute force written here in plain Python from the definition of
  the batch copy (each destination byte inside descriptor i's destination
  range takes the matching source byte; every other byte keeps its value),
  over every batch of one or two descriptors in small pools and over sampled
  three-descriptor batches.
* Invariants on larger random batches: bytes outside the destination ranges
  are untouched, per-descriptor checksums match, permuting the descriptors
  changes nothing, n == 0 is the identity, the copied byte count is the sum
  of the sizes.
* Published FNV-1a test vectors for the checksum.
* An O(n^2) pairwise check for the disjointness test.
* Planted mistakes (a dropped tail, swapped operands, an index off by 8, a
  dropped descriptor) that the pins must catch.
"""

import itertools

import numpy as np
import pytest

import oracle

POOL = 48
OFFSETS = range(0, POOL, 8)
SIZES = (0, 8, 16, 24)


def brute_force(dst_before, src, src_off, dst_off, sizes):
    out = bytearray(dst_before.tobytes())
    for j in range(len(out)):
        for s, d, z in zip(src_off, dst_off, sizes):
            if d <= j < d + z:
                out[j] = src[s + (j - d)]
    return np.frombuffer(bytes(out), dtype=np.uint8)


def _disjoint_pairwise(off, sizes):
    for i in range(len(off)):
        for k in range(i + 1, len(off)):
            if sizes[i] and sizes[k] and off[i] < off[k] + sizes[k] and off[k] < off[i] + sizes[i]:
                return False
    return True


def _all_descriptors():
    for s, d, z in itertools.product(OFFSETS, OFFSETS, SIZES):
        if s + z <= POOL and d + z <= POOL:
            yield (s, d, z)


@pytest.fixture(scope="module")
def tiny_pools():
    g = np.random.default_rng(7)
    src = g.integers(0, 256, POOL, dtype=np.uint8)
    dst = np.full(POOL, 0xA5, dtype=np.uint8)
    return src, dst


def _check_batch(src, dst0, descs, fn=None):
    so = [x[0] for x in descs]
    do = [x[1] for x in descs]
    sz = [x[2] for x in descs]
    want = brute_force(dst0, src, so, do, sz)
    got = dst0.copy()
    (fn or oracle.copy_batch)(got, src, so, do, sz)
    return np.array_equal(got, want)


def test_bruteforce_every_single_and_pair(tiny_pools):
    src, dst0 = tiny_pools
    singles = list(_all_descriptors())
    n_checked = 0
    for a in singles:
        assert _check_batch(src, dst0, [a])
        assert _check_batch(src, dst0, [a], oracle.copy_batch_bytewise)
        n_checked += 1
    for a, b in itertools.combinations(singles, 2):
        if not _disjoint_pairwise([a[1], b[1]], [a[2], b[2]]):
            continue
        assert _check_batch(src, dst0, [a, b]), (a, b)
        n_checked += 1
    assert n_checked > 5000


def test_bruteforce_sampled_triples(tiny_pools):
    src, dst0 = tiny_pools
    singles = list(_all_descriptors())
    g = np.random.default_rng(11)
    done = 0
    while done < 1500:
        idx = g.choice(len(singles), 3, replace=False)
        descs = [singles[i] for i in idx]
        if not _disjoint_pairwise([x[1] for x in descs], [x[2] for x in descs]):
            continue
        assert _check_batch(src, dst0, descs)
        assert _check_batch(src, dst0, descs, oracle.copy_batch_bytewise)
        done += 1


def test_same_pool_copy(tiny_pools):
    src, _ = tiny_pools
    # A copy inside one pool with disjoint source and destination ranges.
    pool = src.copy()
    want = brute_force(pool, pool.copy(), [0, 8], [24, 40], [16, 8])
    oracle.copy_batch(pool, pool, [0, 8], [24, 40], [16, 8])
    assert np.array_equal(pool, want)


def _random_batch(g, pool_bytes, n, max_size):
    """n descriptors with disjoint destination ranges (slot draws), 8-byte granular."""
    slot = max_size
    n_slots = pool_bytes // slot
    dst_slots = g.permutation(n_slots)[:n]
    src_slots = g.integers(0, n_slots, n)
    sizes = 8 * g.integers(0, max_size // 8 + 1, n)
    d_shift = 8 * g.integers(0, (slot - sizes) // 8 + 1)
    s_shift = 8 * g.integers(0, (slot - sizes) // 8 + 1)
    return (src_slots * slot + s_shift).astype(np.uint64), (dst_slots * slot + d_shift).astype(np.uint64), \
        sizes.astype(np.uint64)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_invariants_random_batches(seed):
    g = np.random.default_rng(seed)
    pool_bytes = 1 << 20
    src = g.integers(0, 256, pool_bytes, dtype=np.uint8)
    dst0 = g.integers(0, 256, pool_bytes, dtype=np.uint8)
    so, do, sz = _random_batch(g, pool_bytes, 100, 8192)
    assert oracle.ranges_disjoint(do, sz)
    out = dst0.copy()
    oracle.copy_batch(out, src, so, do, sz)
    # 1. bytes outside every destination range keep their value
    covered = np.zeros(pool_bytes, dtype=bool)
    for d, z in zip(do, sz):
        covered[int(d):int(d + z)] = True
    assert np.array_equal(out[~covered], dst0[~covered])
    # 2. the number of changed-or-covered bytes is the sum of the sizes
    assert int(covered.sum()) == int(sz.sum())
    # 3. per-descriptor checksums of source and destination ranges agree
    assert np.array_equal(oracle.range_checksums(src, so, sz), oracle.range_checksums(out, do, sz))
    # 4. order of descriptors does not matter
    perm = g.permutation(sz.size)
    out2 = dst0.copy()
    oracle.copy_batch(out2, src, so[perm], do[perm], sz[perm])
    assert np.array_equal(out, out2)
    # 5. n == 0 is the identity
    out3 = dst0.copy()
    oracle.copy_batch(out3, src, [], [], [])
    assert np.array_equal(out3, dst0)


def test_fnv1a64_published_vectors(golden):
    vec = golden("fnv1a64_vectors.txt")
    assert len(vec) == 4
    for key, (val,) in vec.items():
        text = key.strip('"').encode()
        assert oracle.fnv1a64(text) == int(val, 16), key


def test_fnv1a64_detects_one_byte_change():
    a = np.arange(4096, dtype=np.uint32).astype(np.uint8)
    b = a.copy()
    b[1234] ^= 1
    assert oracle.fnv1a64(a) != oracle.fnv1a64(b)


def test_ranges_disjoint_vs_pairwise():
    g = np.random.default_rng(5)
    for _ in range(400):
        n = int(g.integers(0, 8))
        off = (8 * g.integers(0, 32, n)).astype(np.uint64)
        sz = (8 * g.integers(0, 6, n)).astype(np.uint64)
        assert oracle.ranges_disjoint(off, sz) == _disjoint_pairwise(list(off), list(sz))


# ---- planted mistakes: each mutant of the oracle must fail a pin ----------

def _mutant_drop_tail(dst, src, so, do, sz):
    oracle.copy_batch(dst, src, so, do, [max(0, z - 8) for z in sz])


def _mutant_swap_operands(dst, src, so, do, sz):
    oracle.copy_batch(dst, src, do, so, sz)


def _mutant_index_off_by_8(dst, src, so, do, sz):
    so2 = [s + 8 if s + z + 8 <= len(src) else s for s, z in zip(so, sz)]
    oracle.copy_batch(dst, src, so2, do, sz)


def _mutant_drop_last(dst, src, so, do, sz):
    oracle.copy_batch(dst, src, so[:-1], do[:-1], sz[:-1])


@pytest.mark.parametrize("mutant", [_mutant_drop_tail, _mutant_swap_operands,
                                    _mutant_index_off_by_8, _mutant_drop_last])
def test_pins_catch_planted_mistakes(tiny_pools, mutant):
    src, dst0 = tiny_pools
    singles = list(_all_descriptors())
    caught = False
    for a, b in itertools.combinations(singles[::7], 2):
        if not _disjoint_pairwise([a[1], b[1]], [a[2], b[2]]):
            continue
        if not _check_batch(src, dst0, [a, b], mutant):
            caught = True
            break
    assert caught, mutant.__name__


# ---- range_checksums: each entry is FNV-1a of exactly its own slice --------
#
# fnv1a64 is pinned by the published vectors above; these tests pin the
# per-range wrapper to it (one slice per entry, each slice's own offset and
# size), so a wrapper that drops or reuses a size, or an offset, fails.

def _checksum_ranges(g, pool_bytes, n):
    off = (8 * g.integers(0, pool_bytes // 8, n)).astype(np.uint64)
    room = pool_bytes - off
    sz = np.minimum((8 * g.integers(0, 96, n)).astype(np.uint64), room)
    sz[::5] = 0  # zero-size ranges among the others
    return off, sz


def test_range_checksums_each_entry_is_its_slice():
    g = np.random.default_rng(11)
    pool = g.integers(0, 256, 1 << 16, dtype=np.uint8)
    off, sz = _checksum_ranges(g, pool.size, 300)
    assert len(set(int(z) for z in sz)) > 20  # many different lengths in one call
    got = oracle.range_checksums(pool, off, sz)
    for i, (o, z) in enumerate(zip(off, sz)):
        assert int(got[i]) == oracle.fnv1a64(pool[int(o):int(o + z)]), i


def test_range_checksums_golden_foobar_and_empty(golden):
    vec = golden("fnv1a64_vectors.txt")
    pool = np.full(64, 0x5A, dtype=np.uint8)
    pool[16:22] = np.frombuffer(b"foobar", dtype=np.uint8)
    pool[40] = ord("a")
    got = oracle.range_checksums(pool, [16, 40, 0, 30], [6, 1, 0, 0])
    assert int(got[0]) == int(vec['"foobar"'][0], 16)
    assert int(got[1]) == int(vec['"a"'][0], 16)
    assert int(got[2]) == int(vec['""'][0], 16)  # an empty range hashes to the offset basis
    assert int(got[3]) == int(vec['""'][0], 16)


def _mutant_checksums_ignore_sizes(pool, off, sz):
    return oracle.range_checksums(pool, off, np.zeros_like(sz))


def _mutant_checksums_first_size(pool, off, sz):
    return oracle.range_checksums(pool, off, np.minimum(np.full_like(sz, sz[0]), pool.size - off))


def _mutant_checksums_first_offset(pool, off, sz):
    return oracle.range_checksums(pool, np.full_like(off, off[0]), np.minimum(sz, pool.size - off[0]))


@pytest.mark.parametrize("mutant", [_mutant_checksums_ignore_sizes, _mutant_checksums_first_size,
                                    _mutant_checksums_first_offset])
def test_range_checksum_pins_catch_planted_mistakes(mutant):
    g = np.random.default_rng(12)
    pool = g.integers(0, 256, 1 << 12, dtype=np.uint8)
    off, sz = _checksum_ranges(g, pool.size, 40)
    bad = mutant(pool, off, sz)
    want = [oracle.fnv1a64(pool[int(o):int(o + z)]) for o, z in zip(off, sz)]
    assert [int(x) for x in bad] != want, mutant.__name__

"""Seeded synthetic inputs for the batched copy: pools, slot draws, descriptor sets.

This module is shared by the oracle-side tests and the GPU side (tests, smoke,
bench). It holds no copy arithmetic at all: it only says which bytes fill
which pool and which (source, destination, size) triples form a batch, as
byte offsets into the pools' bodies. Turning offsets into device or host
addresses, copying and checking happen elsewhere.

Every pool is ``GUARD`` bytes of guard band, then the body, then another guard
band; descriptors address the body only, so a stray write lands in a guard
band that every check compares.

The workloads follow the pages' transfer shapes:

* ``tiny_h2d``: 1,024 x 4 KiB, sources in shuffled slots of an 8 MiB pinned
  host pool, destinations a random permutation of the slots of a 16 MiB
  canary-filled device pool (a small case of the KV transfer shape of PegaFlow
  issue #408, §Test setup / Transfer workload).
* ``kv_burst``: 16,384 shuffled 4 KiB descriptors per direction, 64 MiB H2D +
  64 MiB D2H submitted on two streams, 1 GiB host and device pools (PegaFlow
  issue #408, §Test setup / Transfer workload; follow-up §Setup).
* ``sweep_cell``: descriptor sizes 4-64 KiB around the 28 KiB threshold of the
  vLLM PR #42212 report (§实现拆解 item 2), 8-byte aligned, optionally with
  8-byte granular odd tails and +8 byte starts.
* ``MoeGather``: 6 host banks x 256 experts with the per-expert row bytes of
  FreeToken issue #751 (§Setup: 1,781,760 B per expert in 6 banks) gathered
  into a 3,164-slot device cache, 32 misses per call.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED = 20261202
GUARD = 4096
CANARY = 0xA5
KIB = 1024
MIB = 1024 * 1024
GIB = 1024 * MIB

# FreeToken issue #751, §Setup: 6 banks per expert (gate_up packed/scale/global,
# down packed/scale/global), 1,781,760 bytes per expert in total.
MOE_ROW_BYTES = (1_048_576, 131_072, 4_096, 524_288, 69_632, 4_096)
MOE_EXPERTS = 256
MOE_SLOTS = 3_164
MOE_MISSES_PER_CALL = 32


def rng(*key: int) -> np.random.Generator:
    """A PCG64 generator keyed by (SEED, *key)."""
    return np.random.default_rng([SEED, *[int(k) for k in key]])


@dataclass
class PoolSpec:
    """A byte pool: ``GUARD`` + ``body_bytes`` + ``GUARD``.

    ``where`` is "host" (mapped pinned host memory) or "device" (HBM).
    ``fill`` is "random" (seeded uniform bytes) or "canary" (0xA5 everywhere).
    """
    name: str
    where: str
    body_bytes: int
    fill: str
    seed_key: tuple = ()

    @property
    def total_bytes(self) -> int:
        return self.body_bytes + 2 * GUARD


@dataclass
class Batch:
    """One batch: ``n`` descriptors as offsets into the bodies of two pools."""
    src_pool: str
    dst_pool: str
    src_off: np.ndarray
    dst_off: np.ndarray
    sizes: np.ndarray
    direction: str  # "h2d", "d2h" or "d2d"

    @property
    def n(self) -> int:
        return int(self.sizes.size)

    @property
    def payload_bytes(self) -> int:
        return int(self.sizes.sum(dtype=np.uint64))


@dataclass
class Workload:
    name: str
    pools: dict = field(default_factory=dict)      # name -> PoolSpec
    batches: list = field(default_factory=list)    # list of Batch (or list of lists per step)


def fill_pool(buf: np.ndarray, spec: PoolSpec, block: int = 64 * MIB) -> None:
    """Fill a whole pool buffer (guards included) from its spec, in place."""
    if buf.dtype != np.uint8 or buf.size != spec.total_bytes:
        raise ValueError(f"pool {spec.name}: buffer of {buf.size} bytes, spec wants {spec.total_bytes}")
    if spec.fill == "canary":
        buf.fill(CANARY)
        return
    if spec.fill != "random":
        raise ValueError(f"unknown fill {spec.fill!r}")
    g = rng(*spec.seed_key)
    for a in range(0, buf.size, block):
        b = min(a + block, buf.size)
        buf[a:b] = np.frombuffer(g.bytes(b - a), dtype=np.uint8)


def _u64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint64))


def tiny_h2d() -> Workload:
    """1,024 x 4 KiB H2D into a canary-filled 16 MiB device pool."""
    slot = 4 * KIB
    g = rng(1)
    src_slots = g.permutation(8 * MIB // slot)[:1024]
    dst_slots = g.permutation(16 * MIB // slot)[:1024]
    w = Workload("tiny_h2d: 1,024 x 4 KiB H2D, 8 MiB pinned host pool -> 16 MiB device pool")
    w.pools["host"] = PoolSpec("host", "host", 8 * MIB, "random", (1, 100))
    w.pools["dev"] = PoolSpec("dev", "device", 16 * MIB, "canary")
    w.batches.append(Batch("host", "dev", _u64(src_slots * slot), _u64(dst_slots * slot),
                           _u64(np.full(1024, slot)), "h2d"))
    return w


def kv_burst(n_sets: int = 1, n_per_dir: int = 16_384, pool_bytes: int = GIB) -> Workload:
    """The bidirectional KV burst: per set, one H2D batch and one D2H batch.

    All slots of all sets are distinct on each side, so H2D of any set and D2H
    of any set touch disjoint bytes (safe on two concurrent streams): H2D reads
    host set A_k and writes device set C_k, D2H reads device set D_k and writes
    host set B_k.
    """
    slot = 4 * KIB
    n_slots = pool_bytes // slot
    need = 2 * n_per_dir * n_sets
    if need > n_slots:
        raise ValueError(f"{n_sets} sets of 2 x {n_per_dir} slots do not fit {n_slots} slots")
    g = rng(2, n_per_dir, pool_bytes)
    host_slots = g.permutation(n_slots)[:need].reshape(n_sets, 2, n_per_dir)
    dev_slots = g.permutation(n_slots)[:need].reshape(n_sets, 2, n_per_dir)
    w = Workload(f"kv_burst: {n_per_dir} x 4 KiB per direction, H2D || D2H on two streams, "
                 f"{pool_bytes // MIB} MiB host and device pools")
    # The host pool is random everywhere: set A is read, set B is overwritten.
    w.pools["host"] = PoolSpec("host", "host", pool_bytes, "random", (2, 100))
    w.pools["dev"] = PoolSpec("dev", "device", pool_bytes, "random", (2, 200))
    sizes = _u64(np.full(n_per_dir, slot))
    for k in range(n_sets):
        h2d = Batch("host", "dev", _u64(host_slots[k, 0] * slot), _u64(dev_slots[k, 0] * slot), sizes, "h2d")
        d2h = Batch("dev", "host", _u64(dev_slots[k, 1] * slot), _u64(host_slots[k, 1] * slot), sizes, "d2h")
        w.batches.append((h2d, d2h))
    return w


SWEEP_SIZES_KIB = (4, 8, 12, 16, 24, 28, 32, 64)
SWEEP_COUNTS = (16, 256, 4_096, 65_536)
SWEEP_CAP_BYTES = 512 * MIB


def sweep_cell(size_kib: int, n: int, direction: str, odd_tails: bool = False,
               cap_bytes: int = SWEEP_CAP_BYTES) -> Workload:
    """One cell of the size x count sweep.

    n is capped so that n * size <= cap_bytes. Slots are drawn without
    replacement from pools of 2n slots on each side. With ``odd_tails`` each
    size is ``size - 8*u`` with u odd in [1, 255] (so size mod 16 == 8), and
    the source and destination starts are independently moved by +8 bytes
    with probability 1/2 each; slots are then ``size + 4 KiB`` wide.
    """
    if direction not in ("h2d", "d2h", "d2d"):
        raise ValueError(direction)
    size = size_kib * KIB
    n_eff = max(1, min(n, cap_bytes // size))
    stride = size + (4 * KIB if odd_tails else 0)
    n_slots = 2 * n_eff
    g = rng(3, size_kib, n, {"h2d": 0, "d2h": 1, "d2d": 2}[direction], int(odd_tails))
    src_slots = g.permutation(n_slots)[:n_eff]
    dst_slots = g.permutation(n_slots)[:n_eff]
    src_off = src_slots.astype(np.uint64) * stride
    dst_off = dst_slots.astype(np.uint64) * stride
    if odd_tails:
        u = 2 * g.integers(0, 128, n_eff) + 1            # odd, 1..255
        sizes = (size - 8 * u).astype(np.uint64)
        src_off = src_off + 8 * g.integers(0, 2, n_eff).astype(np.uint64)
        dst_off = dst_off + 8 * g.integers(0, 2, n_eff).astype(np.uint64)
    else:
        sizes = np.full(n_eff, size, dtype=np.uint64)
    src_where = "host" if direction == "h2d" else "device"
    dst_where = "host" if direction == "d2h" else "device"
    tag = "odd" if odd_tails else "aligned"
    w = Workload(f"sweep: {n_eff} x {size_kib} KiB {tag} {direction}")
    w.pools["src"] = PoolSpec("src", src_where, n_slots * stride, "random", (3, size_kib, n, 7))
    w.pools["dst"] = PoolSpec("dst", dst_where, n_slots * stride, "canary")
    w.batches.append(Batch("src", "dst", _u64(src_off), _u64(dst_off), _u64(sizes), direction))
    return w


class MoeGather:
    """MoE expert-miss gather: host banks -> device slot cache, 32 misses per call.

    Host pool: the 6 banks back to back, bank b holding 256 rows of
    ``MOE_ROW_BYTES[b]``. Device pool: the 6 cache arrays back to back, cache
    b holding ``n_slots`` rows of ``MOE_ROW_BYTES[b]``. Expert e of a call is
    placed in one free slot s of every cache array. Each call draws its
    experts uniformly without replacement, and its slots uniformly from the
    slots no earlier call filled (the cache restarts empty when fewer than 32
    remain).
    """

    def __init__(self, n_experts: int = MOE_EXPERTS, n_slots: int = MOE_SLOTS,
                 misses: int = MOE_MISSES_PER_CALL, row_bytes=MOE_ROW_BYTES):
        self.row_bytes = tuple(int(r) for r in row_bytes)
        self.n_experts, self.n_slots, self.misses = n_experts, n_slots, misses
        self.bank_base = np.cumsum((0,) + tuple(r * n_experts for r in self.row_bytes))[:-1]
        self.cache_base = np.cumsum((0,) + tuple(r * n_slots for r in self.row_bytes))[:-1]
        self.pools = {
            "host": PoolSpec("host", "host", sum(self.row_bytes) * n_experts, "random", (4, 100)),
            "dev": PoolSpec("dev", "device", sum(self.row_bytes) * n_slots, "canary"),
        }
        self._g = rng(4, n_experts, n_slots, misses)
        self._free = np.arange(n_slots)

    @property
    def expert_bytes(self) -> int:
        return sum(self.row_bytes)

    def next_call(self) -> Batch:
        g = self._g
        if self._free.size < self.misses:
            self._free = np.arange(self.n_slots)
        experts = g.choice(self.n_experts, self.misses, replace=False)
        pick = g.choice(self._free.size, self.misses, replace=False)
        slots = self._free[pick]
        self._free = np.delete(self._free, pick)
        src, dst, sz = [], [], []
        for e, s in zip(experts, slots):
            for b, r in enumerate(self.row_bytes):
                src.append(self.bank_base[b] + int(e) * r)
                dst.append(self.cache_base[b] + int(s) * r)
                sz.append(r)
        return Batch("host", "dev", _u64(src), _u64(dst), _u64(sz), "h2d")

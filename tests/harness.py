"""Test harness: allocate the workloads' pools, run batches through the C ABI, compare with the oracle.

Host pools are mapped pinned memory from ``kvx_host_alloc``; device pools are
torch uint8 tensors (plumbing only). Expected results come from the oracle
applied to host snapshots of the pools taken before the GPU call; the whole
pool, guard bands included, is compared byte for byte.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W
from expert_host_block_gb300 import kvx


class Pools:
    def __init__(self, specs: dict, device: str = "cuda"):
        self.specs = dict(specs)
        self.bufs = {}
        for name, spec in self.specs.items():
            if spec.where == "host":
                hb = kvx.HostBuffer(spec.total_bytes)
                W.fill_pool(hb.numpy(), spec)
                self.bufs[name] = hb
            else:
                t = torch.empty(spec.total_bytes, dtype=torch.uint8, device=device)
                if spec.fill == "canary":
                    t.fill_(W.CANARY)
                else:
                    host = np.empty(spec.total_bytes, dtype=np.uint8)
                    W.fill_pool(host, spec)
                    t.copy_(torch.from_numpy(host))
                self.bufs[name] = t
        torch.cuda.synchronize()

    def base(self, name: str) -> int:
        """Address of the pool's body (after the leading guard band)."""
        b = self.bufs[name]
        return (b.addr if isinstance(b, kvx.HostBuffer) else b.data_ptr()) + W.GUARD

    def snapshot(self, name: str) -> np.ndarray:
        b = self.bufs[name]
        if isinstance(b, kvx.HostBuffer):
            return b.numpy().copy()
        return b.cpu().numpy()

    def addrs(self, batch: W.Batch):
        return (batch.src_off + np.uint64(self.base(batch.src_pool)),
                batch.dst_off + np.uint64(self.base(batch.dst_pool)), batch.sizes)

    def expected(self, batches) -> dict:
        """Oracle result of running `batches` (all of them, any order) on the current pools."""
        snaps = {name: self.snapshot(name) for name in self.specs}
        want = {name: s.copy() for name, s in snaps.items()}
        g = np.uint64(W.GUARD)
        for b in batches:
            oracle.copy_batch(want[b.dst_pool], snaps[b.src_pool], b.src_off + g, b.dst_off + g, b.sizes)
        return want

    def assert_equal(self, want: dict, names=None) -> None:
        for name in (names or want):
            got = self.snapshot(name)
            if not np.array_equal(got, want[name]):
                bad = np.flatnonzero(got != want[name])
                raise AssertionError(
                    f"pool {name}: {bad.size} bytes differ from the oracle; first at offset "
                    f"{int(bad[0]) - W.GUARD} (body-relative), got {got[bad[0]]:#x} want {want[name][bad[0]]:#x}")

    def close(self):
        for b in self.bufs.values():
            if isinstance(b, kvx.HostBuffer):
                b.close()
        self.bufs.clear()
        torch.cuda.empty_cache()


def run_batch(pools: Pools, batch: W.Batch, stream=None, launch=None, cta_budget=0) -> None:
    s, d, z = pools.addrs(batch)
    if launch is None:
        kvx.kvx_copy_batch(s, d, z, None, batch.direction, cta_budget, stream)
    else:
        kvx.kvx_copy_batch_ex(s, d, z, None, batch.direction, launch, stream)

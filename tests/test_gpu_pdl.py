"""Back-to-back copies launched with programmatic dependent launch stay ordered.

Every copy kernel lets the grid after it on the stream launch early and reads
only its chunk table before it waits for the grid before it. Chains of copies
over pre-uploaded descriptor buffers (no table upload between the kernels, so
each kernel follows the previous one directly on the stream) must then give
exactly what the same hops give one after the other on the CPU: each hop reads
what the previous hop wrote, and later hops overwrite pools that earlier hops
read. The hops mix the LDG kernel by position and from the work counter, the
bulk ring, the staged kernel, and device-resident descriptor lists (plan +
copy kernels), eagerly and as a captured CUDA graph replayed twice. The whole
pools, guard bands included, are compared byte for byte with the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools

pytestmark = pytest.mark.gpu

SLOT = 16 * 1024
N_SLOTS = 4096
BODY = SLOT * N_SLOTS  # 64 MiB per pool


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _hop(g, src, dst, direction, n, aligned):
    if aligned:  # whole 16 KiB slots: the bulk ring's case
        sizes = np.full(n, SLOT, dtype=np.uint64)
        s = (g.permutation(N_SLOTS)[:n] * SLOT).astype(np.uint64)
        d = (g.permutation(N_SLOTS)[:n] * SLOT).astype(np.uint64)
    else:
        sizes = (8 * g.integers(1, 2 * 1024 + 1, n)).astype(np.uint64)  # 8 B .. 16 KiB
        s = (g.permutation(N_SLOTS)[:n] * SLOT + 8 * g.integers(0, 2, n)).astype(np.uint64)
        d = (g.permutation(N_SLOTS)[:n] * SLOT + 8 * g.integers(0, 2, n)).astype(np.uint64)
        sizes = np.minimum(sizes, SLOT - 8).astype(np.uint64)
    return W.Batch(src, dst, s, d, sizes, direction)


# (src pool, dst pool, direction, launch); each hop reads the pool the hop before wrote
HOPS = [
    ("h0", "p0", "h2d", {"variant": "ldg", "assign": "dynamic", "cta_budget": 8}),
    ("p0", "p1", "d2d", {"variant": "ldg"}),
    ("p1", "p2", "d2d", {"variant": "bulk", "cta_budget": 64}),
    ("p2", "p3", "d2d", {"variant": "stage", "cta_budget": 200}),
    ("p3", "p0", "d2d", {"variant": "ldg"}),                    # overwrites what hop 2 read
    ("p0", "h1", "d2h", {"variant": "ldg", "assign": "dynamic", "cta_budget": 4}),
    ("h1", "p1", "h2d", {"variant": "bulk", "cta_budget": 16}),
    ("p1", "h0", "d2h", {"variant": "ldg"}),                    # h0 was the first source
    ("h0", "p2", "h2d", {"variant": "stage", "stages": 2}),
    ("p2", "p3", "d2d", {"variant": "bulk", "cta_budget": 300}),
]


def _specs(seed):
    specs = {"h0": W.PoolSpec("h0", "host", BODY, "random", (93, seed, 0)),
             "h1": W.PoolSpec("h1", "host", BODY, "canary")}
    for k in range(4):
        specs[f"p{k}"] = W.PoolSpec(f"p{k}", "device", BODY, "canary" if k else "random", (93, seed, 2))
    return specs


def _chain(seed):
    g = np.random.default_rng([W.SEED, 93, seed])
    out = []
    for src, dst, direction, launch in HOPS:
        aligned = launch.get("variant") == "bulk"
        n = int(g.choice([64, 700, 2048]))
        out.append((_hop(g, src, dst, direction, n, aligned), launch))
    return out


def _oracle(p, hops):
    want = {name: p.snapshot(name) for name in p.specs}
    gd = np.uint64(W.GUARD)
    for b in hops:
        src = want[b.src_pool].copy()
        oracle.copy_batch(want[b.dst_pool], src, b.src_off + gd, b.dst_off + gd, b.sizes)
    return want


def _bufs(p, chain):
    bufs = []
    for b, _ in chain:
        buf = kvx.DescBuf(int(sum(-(-int(z) // 16384) for z in b.sizes)) + 1)
        buf.upload(*p.addrs(b), b.direction)
        bufs.append(buf)
    torch.cuda.synchronize()
    return bufs


@pytest.mark.parametrize("seed", range(3))
def test_uploaded_chain_back_to_back(seed):
    p = Pools(_specs(seed))
    bufs = []
    try:
        chain = _chain(seed)
        want = _oracle(p, [b for b, _ in chain])
        bufs = _bufs(p, chain)
        s = torch.cuda.Stream()
        for buf, (_, launch) in zip(bufs, chain):
            buf.copy(stream=s, launch=launch)
        kvx.kvx_stream_check(s)
        p.assert_equal(want)
    finally:
        for buf in bufs:
            buf.close()
        p.close()


def test_same_buffer_relaunched_back_to_back():
    # A counter-assigned copy zeroes its table's counter as it ends; the next
    # copy over the same table, launched early, may take units only after that.
    specs = {"h0": W.PoolSpec("h0", "host", BODY, "random", (94,)),
             "p0": W.PoolSpec("p0", "device", BODY, "canary"),
             "p1": W.PoolSpec("p1", "device", BODY, "canary")}
    p = Pools(specs)
    try:
        g = np.random.default_rng([W.SEED, 94])
        a = _hop(g, "h0", "p0", "h2d", 4096, False)   # 4,096 chunks over 4 x 8 warps: counter path
        b = W.Batch("p0", "p1", a.dst_off, a.dst_off, a.sizes, "d2d")
        want = _oracle(p, [a, b, a, b, a, b])
        ba, bb = kvx.DescBuf(4096), kvx.DescBuf(4096)
        ba.upload(*p.addrs(a), "h2d")
        bb.upload(*p.addrs(b), "d2d")
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        la = {"variant": "ldg", "assign": "dynamic", "cta_budget": 4, "threads": 256}
        for _ in range(3):
            ba.copy(stream=s, launch=la)
            ba.copy(stream=s, launch=la)
            bb.copy(stream=s)
        kvx.kvx_stream_check(s)
        p.assert_equal(want)
        ba.close()
        bb.close()
    finally:
        p.close()


def test_uploaded_chain_as_graph_replay():
    p = Pools(_specs(7))
    bufs = []
    try:
        chain = _chain(7)
        hops = [b for b, _ in chain]
        bufs = _bufs(p, chain)
        s = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for buf, (_, launch) in zip(bufs, chain):
                buf.copy(stream=s, launch=launch)
        torch.cuda.synchronize()
        for _ in range(2):  # each replay runs the chain again on the pools as they are
            want = _oracle(p, hops)
            graph.replay()
            torch.cuda.synchronize()
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        for buf in bufs:
            buf.close()
        p.close()


def test_device_list_chain_back_to_back():
    # plan + copy kernels per hop, four hops on one stream, each reading the pool
    # the hop before wrote; the lists live in device memory
    specs = {"p0": W.PoolSpec("p0", "device", BODY, "random", (95,))}
    for k in range(1, 4):
        specs[f"p{k}"] = W.PoolSpec(f"p{k}", "device", BODY, "canary")
    p = Pools(specs)
    lists = []
    try:
        g = np.random.default_rng([W.SEED, 95])
        hops = [_hop(g, f"p{k}", f"p{k + 1}", "d2d", 1500, False) for k in range(3)]
        hops.append(_hop(g, "p3", "p0", "d2d", 1500, False))
        want = _oracle(p, hops)
        dev = []
        for b in hops:
            s_, d_, z_ = p.addrs(b)
            arrs = [torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).cuda() for a in (s_, d_, z_)]
            cnt = torch.full((1,), b.n, dtype=torch.int32, device="cuda")
            dev.append((arrs, cnt))
            lists.append(kvx.DeviceList(b.n))
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        for dl, (arrs, cnt) in zip(lists, dev):
            dl.copy(arrs[0].data_ptr(), arrs[1].data_ptr(), arrs[2].data_ptr(), cnt.data_ptr(), "d2d", stream=s)
        kvx.kvx_stream_check(s)
        p.assert_equal(want)
    finally:
        for dl in lists:
            dl.close()
        p.close()


@pytest.mark.parametrize("variant", ["ldg", "stage", "bulk"])
def test_foreign_kernels_around_copies(variant):
    # PyTorch kernels (launched without programmatic serialisation) write a copy's
    # source right before it and read its destination right after it, on the same
    # stream with no synchronisation: each must still see the other's bytes.
    n, size = 2048, 16384
    src = torch.zeros(n * size // 4, dtype=torch.int32, device="cuda")
    mid = torch.zeros_like(src)
    out = torch.zeros_like(src)
    g = np.random.default_rng([W.SEED, 97])
    perm = g.permutation(n).astype(np.uint64)
    z = np.full(n, size, dtype=np.uint64)
    off = np.arange(n, dtype=np.uint64) * np.uint64(size)
    a = kvx.DescBuf(n)  # src -> mid, blocks permuted
    b = kvx.DescBuf(n)  # mid -> out, back in order
    a.upload(np.uint64(src.data_ptr()) + off, np.uint64(mid.data_ptr()) + perm * np.uint64(size), z, "d2d")
    b.upload(np.uint64(mid.data_ptr()) + perm * np.uint64(size), np.uint64(out.data_ptr()) + off, z, "d2d")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    launch = {"variant": variant}
    try:
        with torch.cuda.stream(s):
            for step in range(1, 6):
                src.fill_(step)                  # torch writes the source
                a.copy(stream=s, launch=launch)  # kvx copies it
                mid.add_(10)                     # torch rewrites the copy's output in place
                b.copy(stream=s, launch=launch)
                out.mul_(2)                      # torch reads and writes the second copy's output
        kvx.kvx_stream_check(s)
        assert torch.all(out == 2 * (5 + 10)).item()
        assert torch.all(mid == 5 + 10).item()
    finally:
        a.close()
        b.close()


def test_chain_with_programmatic_launch_off():
    # KVX_PDL=0: the same kernels launched without the attribute (plain stream order); a chain of
    # uploaded copies and the smoke batch still match the oracle
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys\n"
            "sys.path.insert(0, 'tests')\n"
            "import __graft_entry__ as g\n"
            "g.smoke()\n"
            "import test_gpu_pdl as t\n"  # smoke() has built the library and selected cuda:0
            "t.test_uploaded_chain_back_to_back(1)\n"
            "print('chain ok')\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=root,
                         env=dict(os.environ, KVX_PDL="0"))
    assert out.returncode == 0 and "smoke ok" in out.stdout and "chain ok" in out.stdout, out.stdout + out.stderr

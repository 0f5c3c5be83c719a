"""MoE expert-miss gathers at adversarial miss counts, boundary experts and boundary slots.

The FreeToken page verified its gather byte-exact over many calls, with
adversarial cases of 0 to hundreds of misses, boundary slots and experts, in
eager mode and in graph replay (FreeToken issue #751, §Correctness evidence).
Here: miss counts 0, 1, 31, 32, 33, 255 and 256 (every expert of a layer),
each including the first and last expert and the first and last cache slot
where the count allows, through kvx_copy_batch and through one captured
device-list copy replayed with each list; every call is compared with the
oracle over the whole device cache.
"""

import numpy as np
import pytest
import torch

import workloads as W
from expert_host_block_gb300 import kvx
from harness import Pools

pytestmark = pytest.mark.gpu

COUNTS = [0, 1, 31, 32, 33, 255, 256]
N_SLOTS = 600


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from expert_host_block_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _call(m, experts, slots):
    src, dst, sz = [], [], []
    for e, s in zip(experts, slots):
        for b, r in enumerate(m.row_bytes):
            src.append(m.bank_base[b] + int(e) * r)
            dst.append(m.cache_base[b] + int(s) * r)
            sz.append(r)
    u = lambda a: np.asarray(a, dtype=np.uint64)
    return W.Batch("host", "dev", u(src), u(dst), u(sz), "h2d")


def _with_ends(n, count, g):
    """`count` distinct values of range(n), the first and last of them included when count >= 2."""
    if count == 0:
        return np.zeros(0, dtype=np.int64)
    if count == 1:
        return np.array([n - 1])
    rest = 1 + g.permutation(n - 2)[: count - 2]  # from 1 .. n - 2
    return np.concatenate([[0, n - 1], rest])


def _adversarial(m, count, g):
    experts = _with_ends(m.n_experts, count, g)
    slots = _with_ends(m.n_slots, count, g)
    assert len(set(experts.tolist())) == count and len(set(slots.tolist())) == count
    return _call(m, experts, slots)


def test_moe_adversarial_counts_eager():
    m = W.MoeGather(n_slots=N_SLOTS)
    p = Pools(m.pools)
    g = np.random.default_rng([W.SEED, 97])
    try:
        for count in COUNTS:
            b = _adversarial(m, count, g)
            want = p.expected([b])
            kvx.kvx_copy_batch(*p.addrs(b), None, "h2d", 0, None)
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        p.close()


def test_moe_adversarial_counts_graph_replay():
    m = W.MoeGather(n_slots=N_SLOTS)
    p = Pools(m.pools)
    g = np.random.default_rng([W.SEED, 98])
    max_n = 256 * len(m.row_bytes)
    lst = kvx.DeviceList(max_n)
    arr = [torch.zeros(max_n, dtype=torch.int64, device="cuda") for _ in range(3)]
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    gs = torch.cuda.Stream()
    try:
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            lst.copy(*(a.data_ptr() for a in arr), cnt.data_ptr(), "h2d", stream=gs)
        for count in COUNTS:
            b = _adversarial(m, count, g)
            want = p.expected([b])
            s, d, z = p.addrs(b)
            for a, v in zip(arr, (s, d, z)):
                a.zero_()
                if v.size:
                    a[: v.size].copy_(torch.from_numpy(v.view(np.int64)))
            cnt.fill_(b.n)
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            kvx.kvx_stream_check(None)
            p.assert_equal(want)
    finally:
        lst.close()
        p.close()

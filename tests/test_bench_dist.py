"""The replica bookkeeping of bench.py on CPU: 2 gloo ranks, no GPU.

kvx shards as independent replicas (one engine per GPU, no data-path
collective). bench.py only reduces two scalars over ranks: the units moved
(sum) and the timed seconds (max). These tests run that path with world
size 2 on the gloo backend, plus the reference arm's rank handling.
"""

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    total, slowest, thr = bench.aggregate(float(rank + 1) * 100.0, float(rank + 1), d)
    d.barrier()
    d.close()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"total": total, "slowest": slowest, "thr": thr}, f)


def test_aggregate_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert res["total"] == pytest.approx(300.0)   # 100 + 200 units over the ranks
        assert res["slowest"] == pytest.approx(2.0)   # max over ranks
        assert res["thr"] == pytest.approx(150.0)


def _ref_rank(rank, world, port, out_dir):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    d = bench.Dist()
    d.init("gloo")

    class A:
        steps, warmup = 1, 0
    import workloads as W
    real = W.kv_burst
    W.kv_burst = lambda n_sets=1: real(n_sets=1, n_per_dir=64, pool_bytes=W.MIB)
    try:
        res = bench.bench_reference(A, d)
    finally:
        W.kv_burst = real
    d.close()
    with open(os.path.join(out_dir, f"ref{rank}.json"), "w") as f:
        json.dump(res, f)


def test_reference_arm_runs_on_rank0_only(tmp_path):
    port = _free_port()
    mp.start_processes(_ref_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0 = json.load(open(tmp_path / "ref0.json"))
    r1 = json.load(open(tmp_path / "ref1.json"))
    assert r1 is None
    assert r0["impl"] == "reference" and r0["value"] > 0 and r0["n_gpus"] == 2
    assert r0["cpu_baseline"]["kind"] == "oracle" and r0["e2e"]["h2d_bytes_per_step"] == 0


def test_single_process_aggregate_is_identity():
    d = bench.Dist()
    assert bench.aggregate(10.0, 2.0, d) == (10.0, 2.0, 5.0)


def test_clock_sampler_without_nvml_reports_why():
    c = bench.ClockSampler(0)
    c.start()
    c.stop()
    s = c.summary()
    if c.error:
        assert s["samples"] == 0 and "NVML" in s["note"]
    else:  # a machine with a GPU
        assert s["samples"] >= 2


def test_parse_cell_specs():
    assert bench.parse_cell("h2d:4:65536") == ("h2d", 4, 65536, False)
    assert bench.parse_cell("d2d:28:4096:odd") == ("d2d", 28, 4096, True)
    for bad in ("x2y:4:16", "h2d:4", "h2d:4:16:even", "d2h:4:16:odd:1"):
        with pytest.raises(SystemExit):
            bench.parse_cell(bad)


def test_graded_passes_rotate_and_take_medians():
    specs = bench.graded_specs()
    seen_first = set()
    for r in range(bench.GRADED_ROUNDS):
        order = bench.rotated(specs, r, bench.GRADED_ROUNDS)
        assert sorted(order) == sorted(specs)  # every cell once per pass
        seen_first.add(order[0])
    assert len(seen_first) == bench.GRADED_ROUNDS  # each pass starts elsewhere
    base = {"dir": "h2d", "size_kib": 4, "n": 4096, "odd": False, "kernel_gbs_best": 0.0}
    rounds = [dict(base, **{k: v for k in bench.ROUND_FIELDS}, kernel_gbs_best=v) for v in (0.9, 0.5, 0.8)]
    rounds[1]["frac_stream"] = None  # a figure missing from one pass
    c = bench.median_of_rounds(rounds)
    assert c["frac"] == c["kernel_gbs"] == 0.8  # one disturbed pass does not move the cell
    assert c["frac_stream"] == pytest.approx(0.85)  # median of the passes that have it
    assert c["kernel_gbs_best"] == 0.9 and c["rounds"] == 3 and c["dir"] == "h2d"

"""The benchmark's multi-process host logic on CPU: two gloo ranks agree on
the slowest rank's time and on the total, and reduce disjoint simulated ranks
(weak scaling: every GPU gets its own seeds)."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        mx = bench.max_over_ranks(10.0 + 5.0 * r, w)
        sm = bench.sum_over_ranks(1.0 + r, w)
        seeds = bench.simulated_ranks(r)
        gathered = [None] * w
        dist.all_gather_object(gathered, seeds)
        q.put((r, w, lr, mx, sm, gathered))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, lr, mx, sm, gathered in out:
        assert w == world and lr == r
        assert mx == 15.0  # the slowest rank's time
        assert sm == 3.0
        flat = [s for g in gathered for s in g]
        assert len(flat) == len(set(flat)) == world * 8  # disjoint seeds per GPU (8 simulated ranks each)


def test_single_process_defaults(monkeypatch):
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.simulated_ranks(0) == list(range(8))
    assert bench.simulated_ranks(3) == list(range(24, 32))


def test_kernel_source_hash_ignores_comments():
    import bench

    code = "int f(int x) {  // doubles\n    return 2 * x;\n}\n"
    assert bench.code_lines(code) == ["int f(int x) {", "    return 2 * x;", "}"]
    assert bench.code_lines("// only a comment\n\n   \n") == []
    assert bench.code_lines(code) == bench.code_lines("// header\n" + code.replace("doubles", "twice"))
    assert bench.code_lines(code) != bench.code_lines(code.replace("2 * x", "3 * x"))


def test_recorded_traffic_is_consistent():
    import json
    import os

    import bench

    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    for k in ("compress_kernel", "reduce_kernel", "decompress_kernel"):
        rec = recs[k]
        want = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) * rec["scale_to_bench_launch"]
        assert abs(rec["bytes_per_launch_scaled"] - want) <= 1e-5 * want
        assert len(rec["source_hash"]) == 16
        # used only while it names the current kernel code
        assert (bench.recorded_traffic(k) is not None) == (rec["source_hash"] == bench.kernel_source_hash())


def test_clock_summary_reads_the_window():
    """The clock record of the line: median SM clock, the maximum, the union
    of clock event reasons and the power, over the samples inside the window
    only; with no GPU the sampler says why it has no samples."""
    import bench

    cs = bench.ClockSampler(0)
    assert cs.nvml is None and cs.note  # no GPU here: the reason is recorded
    cs.samples = [(10.0, 1000.0, 2070.0, set(), 100.0), (11.0, 2070.0, 2070.0, {"sw_power_cap"}, 900.0),
                  (12.0, 2000.0, 2070.0, set(), 800.0), (13.0, 500.0, 2070.0, {"hw_slowdown"}, 50.0)]
    s = cs.summary(10.5, 12.5)
    assert s["samples"] == 2 and s["sm_mhz"] == 2035.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 900.0
    assert cs.summary(20.0, 30.0)["samples"] == 0

"""Benchmark of the compressed data-parallel reduce step on GB300.

One step = the whole hot path over one batch of synthetic input: the 64 MiB
gradient-like bf16 buffer (33,554,432 values ~ N(0, 1e-3), 1% of positions
x100) of R = 2 simulated data-parallel ranks held in this GPU's memory:
    compress(rank 0), compress(rank 1)            split, exponent table, look-back placement
    fused reduce(stream 0, stream 1)              decompress -> binary32 sum -> bf16 -> compress
    decompress(reduced stream)                    the receiver's decode
`value` = uncompressed gradient bytes entering the step (R * 2n) / step time,
timed on the device with CUDA events around each step, the step replayed as
one captured CUDA graph of the four library calls, L2 flushed (256 MiB write,
untimed) before every step, max over ranks.  The ops are timed one by one in
a second pass of plain launches.  N GPUs under torchrun run N independent replicas
(weak scaling); nothing crosses GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]
"""

from __future__ import annotations

import argparse
import hashlib
import platform
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compress / decompress / fused-reduce uncompressed GB/s and % of HBM roofline; ratio"
WORKLOAD = 2          # the 64 MiB gradient-like buffer
RANKS_PER_GPU = 2     # simulated data-parallel ranks reduced on each GPU
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["cccl_device.cuh", "cccl_encode.cuh", "cccl_decode.cuh", "cccl_compress.cu",
                  "cccl_decompress.cu", "cccl_reduce.cu"]


# ---------------------------------------------------------------- host logic (also tested on CPU with gloo)
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def simulated_ranks(gpu_rank: int) -> list[int]:
    """Seeds (rank ids of the workload) reduced by one GPU: disjoint across GPUs."""
    return [RANKS_PER_GPU * gpu_rank + j for j in range(RANKS_PER_GPU)]


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def code_lines(text: str) -> list[str]:
    """The lines of a kernel source that the compiler sees as code: `//`
    comments, trailing blanks and empty lines dropped (no string literal in
    these sources holds `//`)."""
    out = []
    for line in text.splitlines():
        line = line.split("//", 1)[0].rstrip()
        if line:
            out.append(line)
    return out


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code, so that a comment edit does not
    invalidate counters taken on the same code."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "compression_coupled_collectives_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update("\n".join(code_lines(fh.read())).encode())
            h.update(b"\0")
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        sm, smax, reasons = [], [], set()
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- the oracle as a CPU baseline
def oracle_step_seconds(xs, chunks: int) -> tuple[float, int]:
    """Time the oracle doing the step on the first `chunks` chunks of each rank."""
    import oracle

    n = min(xs[0].size, chunks * 4096)
    part = [x[:n] for x in xs]
    t = time.perf_counter()
    streams = [oracle.compress(p) for p in part]
    red = oracle.reduce(streams, n)
    oracle.decompress(red, n)
    return time.perf_counter() - t, n


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else implementer/part)."""
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model", "Hardware"):
        for line in text.splitlines():
            if line.split(":")[0].strip() == key:
                return line.split(":", 1)[1].strip()
    fields = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = (t.strip() for t in line.split(":", 1))
            fields.setdefault(k, v)
    return "%s CPU implementer %s part %s" % (platform.machine(), fields.get("CPU implementer", "?"),
                                              fields.get("CPU part", "?"))


def cpu_baseline_all_cores(xs, budget_s: float = 6.0) -> dict:
    """The oracle, as it stands, on every host core at once: each thread runs
    the step on its own slice of chunks (the oracle is single-threaded C; the
    threads share nothing)."""
    import concurrent.futures as cf

    import oracle

    oracle.build()
    cores = max(1, os.cpu_count() or 1)
    n_chunks = xs[0].size // 4096
    per = max(1, n_chunks // cores)
    probe_t, _ = oracle_step_seconds(xs, 16)
    # chunks per thread so that one round takes about budget_s / 2
    take = max(1, min(per, int(budget_s / 2 / (probe_t / 16))))

    def one(i):
        a = (i * per) * 4096
        part = [x[a:a + take * 4096] for x in xs]
        return oracle_step_seconds(part, take)

    total_n, t0 = 0, time.perf_counter()
    rounds = 0
    with cf.ThreadPoolExecutor(cores) as ex:
        while time.perf_counter() - t0 < budget_s and rounds < 4:
            total_n += sum(n for _, n in ex.map(one, range(cores)))
            rounds += 1
    total_t = time.perf_counter() - t0
    gbs = len(xs) * 2 * total_n / total_t / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": "%d threads, each the full step on its own %d-chunk slice of every rank, %d round(s), %.1f s"
                      % (cores, take, rounds, total_t)}


def cpu_baseline(xs, budget_s: float = 12.0) -> dict:
    import oracle

    oracle.build()
    n_full = xs[0].size
    total_t, total_n, reps = 0.0, 0, 0
    chunks = n_full // 4096
    while total_t < budget_s and reps < 8:
        dt, n = oracle_step_seconds(xs, chunks)
        total_t += dt
        total_n += n
        reps += 1
    gbs = len(xs) * 2 * total_n / total_t / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
            "sample": "the full step on the whole workload (%d ranks x %d values), %d repetition(s), "
                      "%.1f s, single-threaded C oracle" % (len(xs), n_full, reps, total_t)}


def run_reference(args, rank: int, world: int) -> None:
    """The reference arm: the CPU oracle, as it stands, on this host's cores."""
    import numpy as np  # noqa: F401

    import oracle
    import workloads

    oracle.build()
    workloads.build()
    if rank != 0:
        return
    n = workloads.SIZES[WORKLOAD]
    xs = [workloads.generate(WORKLOAD, r) for r in simulated_ranks(0)]
    steps, warmup = args.steps, max(args.warmup, 3)
    # each step: a bounded sample of chunks, rotating through the workload, so
    # that the whole run stays within about two minutes
    per_step_s = 100.0 / (steps + warmup)
    probe_t, probe_n = oracle_step_seconds(xs, 64)
    chunks = max(1, min(n // 4096, int(per_step_s / (probe_t / 64))))
    offs = 0
    total_t, total_n = 0.0, 0
    for i in range(warmup + steps):
        a = (offs % (n // 4096)) * 4096
        b = min(n, a + chunks * 4096)
        part = [x[a:b] for x in xs]
        t = time.perf_counter()
        streams = [oracle.compress(p) for p in part]
        red = oracle.reduce(streams, b - a)
        oracle.decompress(red, b - a)
        dt = time.perf_counter() - t
        offs += chunks
        if i >= warmup:
            total_t += dt
            total_n += b - a
    value = RANKS_PER_GPU * 2 * total_n / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(1e3 * total_t / steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8+f32",
        "data": "synthetic", "config": workload_config(),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "%d chunks of each rank per step, rotating through the workload" % chunks},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config() -> dict:
    return {"workload": "gradient-like bf16 buffer, 33,554,432 values (64 MiB) ~ N(0, 1e-3) with 1%% of "
                        "positions x100, on %d simulated data-parallel ranks per GPU: compress each, fused "
                        "reduce (R=%d), decompress the result" % (RANKS_PER_GPU, RANKS_PER_GPU),
            "n_elems": 33554432, "ranks_per_gpu": RANKS_PER_GPU, "chunk_elems": 4096,
            "l2": "flushed before every timed step (256 MiB write, untimed)",
            "parallelism": "replicas (weak scaling, no cross-GPU traffic)"}


# ---------------------------------------------------------------- rows beyond the step
KV_BLOCK = 16 * 8 * 128  # 16 tokens x 8 heads x 128 dim


def measure_extras(cc, torch, np, xs, streams, sizes, n, flush, peak, reps: int = 50) -> dict:
    """The selective-compression reduce and the paged payload, each timed alone
    (CUDA events on the current stream, L2 flushed before every repetition,
    median), with their algorithmic HBM bytes."""
    import workloads

    stream = torch.cuda.current_stream()
    out = {}

    def timed(fn):
        ts = []
        for k in range(reps + 3):
            flush.fill_(k & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if k >= 3:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    # local rank-0 buffer + one compressed remote rank, 64 MiB each
    red = cc.empty_stream(n)
    ws = cc.empty_workspace(n)
    ms = timed(lambda: cc.cccl_reduce_mixed(xs[0], [streams[1][:sizes[1]]], red, ws, stream=stream))
    out_bytes, st = cc.cccl_get_result(ws, stream)
    algo = 2 * n + sizes[1] + out_bytes
    out["reduce_mixed"] = {"ms": round(ms, 5), "workload": "local rank-0 buffer (uncompressed) + 1 compressed remote "
                           "rank of the 64 MiB gradient-like buffer", "status": st,
                           "uncompressed_gbs": round(2 * 2 * n / (ms * 1e-3) / 1e9, 1), "algorithmic_bytes": algo,
                           "hbm_gbs": round(algo / (ms * 1e-3) / 1e9, 1),
                           "frac_of_measured_copy": round(algo / (ms * 1e-3) / 1e9 / peak, 4)}
    # KV-cache blocks of the [32, 2, 4096, 8, 128] shape: 4096 of a pool of 8192 blocks, shuffled
    n_pool, n_blk = 8192, 4096
    pool = torch.from_numpy(workloads.generate(4, 0, count=n_pool * KV_BLOCK).view(np.int16)).cuda()
    table = torch.from_numpy(np.random.default_rng(7).permutation(n_pool)[:n_blk].astype(np.int32)).cuda()
    npg = n_blk * KV_BLOCK
    s_pg = cc.empty_stream(npg)
    ws_pg = cc.empty_workspace(npg)
    ms_c = timed(lambda: cc.cccl_compress_paged(pool, KV_BLOCK, table, s_pg, ws_pg, stream=stream))
    pbytes, st_c = cc.cccl_get_result(ws_pg, stream)
    target = torch.empty_like(pool)
    ms_d = timed(lambda: cc.cccl_decompress_paged(s_pg[:pbytes], target, KV_BLOCK, table, ws_pg, stream=stream))
    _, st_d = cc.cccl_get_result(ws_pg, stream)
    ok = bool(torch.equal(target.view(n_pool, KV_BLOCK)[table.long()], pool.view(n_pool, KV_BLOCK)[table.long()]))
    for name, ms_x, st_x in (("compress_paged", ms_c, st_c), ("decompress_paged", ms_d, st_d)):
        algo = 2 * npg + pbytes
        out[name] = {"ms": round(ms_x, 5), "workload": "4096 KV-cache blocks of 16 tokens x 8 heads x 128 dim "
                     "(64 Mi values) gathered through a shuffled block table from a pool of 8192", "status": st_x,
                     "uncompressed_gbs": round(2 * npg / (ms_x * 1e-3) / 1e9, 1), "algorithmic_bytes": algo,
                     "hbm_gbs": round(algo / (ms_x * 1e-3) / 1e9, 1),
                     "frac_of_measured_copy": round(algo / (ms_x * 1e-3) / 1e9 / peak, 4),
                     "ratio": round(pbytes / (2 * npg), 5)}
    out["decompress_paged"]["round_trip_exact"] = ok
    # window-base variant (stream version 2) next to the minimum-base stream
    for name, x in (("compress_window", xs[0]),
                    ("compress_window_specials",
                     torch.from_numpy(workloads.generate(5, 0, start=1 << 27, count=n).view(np.int16)).cuda())):
        s_w = cc.empty_stream(n)
        ws_w = cc.empty_workspace(n)
        ms_w = timed(lambda: cc.cccl_compress_window(x, s_w, ws_w, stream=stream))
        wbytes, st_w = cc.cccl_get_result(ws_w, stream)
        cc.cccl_compress(x, s_w, ws_w, stream=stream)
        v1bytes, _ = cc.cccl_get_result(ws_w, stream)
        algo = 2 * n + wbytes
        out[name] = {"ms": round(ms_w, 5), "workload": "64 MiB gradient-like buffer" if name == "compress_window"
                     else "64 MiB of N(0, 1) with 0.1% each NaN, +-Inf, +-0, subnormals (second half of the worst-case "
                     "buffer)", "status": st_w, "uncompressed_gbs": round(2 * n / (ms_w * 1e-3) / 1e9, 1),
                     "algorithmic_bytes": algo, "hbm_gbs": round(algo / (ms_w * 1e-3) / 1e9, 1),
                     "frac_of_measured_copy": round(algo / (ms_w * 1e-3) / 1e9 / peak, 4),
                     "ratio": round(wbytes / (2 * n), 5), "ratio_min_base": round(v1bytes / (2 * n), 5)}
    out.update(measure_dtypes(cc, torch, np, n, timed, stream, peak))
    out.update(measure_workloads(cc, torch, np, timed, stream, peak))
    return out


def measure_workloads(cc, torch, np, timed, stream, peak) -> dict:
    """The larger bf16 workloads at their full sizes, each op timed alone:
    the R=8 fused reduce over 8 x 256 MiB pre-compressed ranks; the 512 MiB
    KV-cache tensor round trip; the 512 MiB worst case (half incompressible)
    round trip and its R=4 fused reduce.  Inputs are far larger than the L2."""
    import workloads

    out = {}
    n_chunks = lambda n: -(-n // 4096)

    def row(ms_x, algo, uncompressed, **kw):
        d = {"ms": round(ms_x, 5), "algorithmic_bytes": int(algo),
             "uncompressed_gbs": round(uncompressed / (ms_x * 1e-3) / 1e9, 1),
             "hbm_gbs": round(algo / (ms_x * 1e-3) / 1e9, 1),
             "frac_of_measured_copy": round(algo / (ms_x * 1e-3) / 1e9 / peak, 4)}
        d.update(kw)
        return d

    def compressed(w, ranks):
        n = workloads.SIZES[w]
        ss, sizes = [], []
        ws = cc.empty_workspace(n)
        for r in range(ranks):
            x = torch.from_numpy(workloads.generate(w, r).view(np.int16)).cuda()
            s_ = cc.empty_stream(n)
            cc.cccl_compress(x, s_, ws, stream=stream)
            b, st = cc.cccl_get_result(ws, stream)
            if st != 0:
                raise RuntimeError("compress of workload %d rank %d: status %d" % (w, r, st))
            ss.append(s_)
            sizes.append(b)
            if r > 0:
                del x
            else:
                x0 = x
        return n, x0, ss, sizes, ws

    def reduce_row(n, ss, sizes, ws, R):
        red = cc.empty_stream(n)
        ins = [s_[:b] for s_, b in zip(ss[:R], sizes[:R])]
        ms_r = timed(lambda: cc.cccl_reduce_compressed(ins, n, red, ws, stream=stream))
        rbytes, st = cc.cccl_get_result(ws, stream)
        tab = 8 * n_chunks(n)
        return row(ms_r, sum(sizes[:R]) + R * tab + rbytes + tab, R * 2 * n, status=st,
                   ratio_out=round(rbytes / (2 * n), 5))

    def round_trip_rows(n, x, s_, b, ws):
        ms_c = timed(lambda: cc.cccl_compress(x, s_, ws, stream=stream))
        _, st_c = cc.cccl_get_result(ws, stream)
        y = torch.empty_like(x)
        ms_d = timed(lambda: cc.cccl_decompress(s_[:b], y, ws, stream=stream))
        _, st_d = cc.cccl_get_result(ws, stream)
        tab = 8 * n_chunks(n)
        return (row(ms_c, 2 * n + b + tab, 2 * n, status=st_c, ratio=round(b / (2 * n), 5)),
                row(ms_d, b + tab + 2 * n, 2 * n, status=st_d, round_trip_exact=bool(torch.equal(x, y))))

    # R = 8 ranks of 134,217,728 values ~ N(0, 0.02)
    n, x0, ss, sizes, ws = compressed(3, 8)
    out["workload3_reduce_r8"] = reduce_row(n, ss, sizes, ws, 8)
    out["workload3_reduce_r8"]["workload"] = "8 pre-compressed ranks of 134,217,728 bf16 values (256 MiB each) " \
                                             "~ N(0, 0.02), fused reduce in rank order 0..7"
    del x0, ss, ws
    # KV-cache tensor [32, 2, 4096, 8, 128]
    n, x0, ss, sizes, ws = compressed(4, 1)
    c_row, d_row = round_trip_rows(n, x0, ss[0], sizes[0], ws)
    kv = "KV-cache tensor [32, 2, 4096, 8, 128] = 268,435,456 bf16 values (512 MiB), per-head log-uniform scales"
    out["workload4_compress"] = dict(c_row, workload=kv)
    out["workload4_decompress"] = dict(d_row, workload=kv)
    del x0, ss, ws
    # worst case: half uniform 16-bit patterns, half N(0, 1) with specials; 4 ranks
    n, x0, ss, sizes, ws = compressed(5, 4)
    c_row, d_row = round_trip_rows(n, x0, ss[0], sizes[0], ws)
    wc = "worst case, 268,435,456 bf16 values (512 MiB): half uniform 16-bit patterns, half N(0, 1) with 0.1% " \
         "each NaN, +-Inf, +-0, subnormals"
    out["workload5_compress"] = dict(c_row, workload=wc)
    out["workload5_decompress"] = dict(d_row, workload=wc)
    out["workload5_reduce_r4"] = dict(reduce_row(n, ss, sizes, ws, 4), workload=wc + "; 4 ranks, fused reduce")
    del x0, ss, ws
    torch.cuda.empty_cache()
    return out


def measure_dtypes(cc, torch, np, n, timed, stream, peak) -> dict:
    """The step (2 x compress, fused sum reduce, decompress of the result) on
    the same gradient-like recipe in fp16 and fp32 (n values per rank), each
    op timed alone, with its algorithmic HBM bytes."""
    import workloads

    out = {}
    for name, dtype, bits in (("fp16", cc.CCCL_DTYPE_FP16, torch.int16), ("fp32", cc.CCCL_DTYPE_FP32, torch.int32)):
        item = 2 if dtype == cc.CCCL_DTYPE_FP16 else 4
        xs = [torch.from_numpy(workloads.generate_typed(dtype, WORKLOAD, r).view(np.int16 if item == 2 else np.int32))
              .cuda() for r in range(2)]
        cap = cc.cccl_compress_bound_typed(dtype, n)
        ss = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in xs]
        ws = cc.empty_workspace(n)
        sizes = []
        for x, s_ in zip(xs, ss):
            cc.cccl_compress_typed(dtype, x, s_, ws, stream=stream)
            sizes.append(cc.cccl_get_result(ws, stream)[0])
        ms_c = timed(lambda: cc.cccl_compress_typed(dtype, xs[0], ss[0], ws, stream=stream))
        red = torch.empty(cap, dtype=torch.uint8, device="cuda")
        ins = [s_[:b] for s_, b in zip(ss, sizes)]
        ms_r = timed(lambda: cc.cccl_reduce_typed(dtype, 0, None, ins, n, red, ws, stream=stream))
        rbytes, st_r = cc.cccl_get_result(ws, stream)
        y = torch.empty(n, dtype=bits, device="cuda")
        ms_d = timed(lambda: cc.cccl_decompress_typed(dtype, red[:rbytes], y, ws, stream=stream))
        _, st_d = cc.cccl_get_result(ws, stream)
        rows = {"compress": (ms_c, item * n + sizes[0]), "reduce": (ms_r, sum(sizes) + rbytes),
                "decompress": (ms_d, rbytes + item * n)}
        entry = {"workload": "gradient-like buffer, %d values per rank (%d MiB of %s), 2 ranks"
                             % (n, item * n >> 20, name), "ratio": round(sizes[0] / (item * n), 5),
                 "status": max(st_r, st_d), "step_ms": round(2 * ms_c + ms_r + ms_d, 5),
                 "step_uncompressed_gbs": round(2 * item * n / ((2 * ms_c + ms_r + ms_d) * 1e-3) / 1e9, 1)}
        for op, (ms_x, algo) in rows.items():
            entry[op] = {"ms": round(ms_x, 5), "algorithmic_bytes": int(algo),
                         "hbm_gbs": round(algo / (ms_x * 1e-3) / 1e9, 1),
                         "frac_of_measured_copy": round(algo / (ms_x * 1e-3) / 1e9 / peak, 4)}
        out["dtype_" + name] = entry
        del xs, ss, red, y
    return out


# ---------------------------------------------------------------- the GPU arm
def run_gpu(args, rank: int, world: int, local_rank: int) -> None:
    import numpy as np
    import torch

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    import __graft_entry__

    __graft_entry__.build()
    import compression_coupled_collectives_gb300 as cc
    import workloads

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)

    seeds = simulated_ranks(rank)
    xs_host = [workloads.generate(WORKLOAD, r) for r in seeds]
    n = xs_host[0].size
    R = len(xs_host)
    pinned = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_host]
    xs = [p.to(device) for p in pinned]
    cap = cc.cccl_compress_bound(n)
    streams = [torch.empty(cap, dtype=torch.uint8, device=device) for _ in range(R)]
    red = torch.empty(cap, dtype=torch.uint8, device=device)
    y = torch.empty(n, dtype=torch.int16, device=device)
    y_host = torch.empty(n, dtype=torch.int16).pin_memory()
    wsb = cc.cccl_workspace_bytes(n)
    ws = [torch.empty(wsb, dtype=torch.uint8, device=device) for _ in range(R + 2)]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(ev=None, s=stream):
        # ev: list of (start, end) event pairs, one per op
        for r in range(R):
            if ev is not None:
                ev[r][0].record(s)
            cc.cccl_compress(xs[r], streams[r], ws[r], s)
            if ev is not None:
                ev[r][1].record(s)
        if ev is not None:
            ev[R][0].record(s)
        cc.cccl_reduce_compressed(streams, n, red, ws[R], stream=s)
        if ev is not None:
            ev[R][1].record(s)
            ev[R + 1][0].record(s)
        cc.cccl_decompress(red, y, ws[R + 1], stream=s)
        if ev is not None:
            ev[R + 1][1].record(s)

    # one untimed pass: sizes, ratios and a sampled check against the oracle
    step()
    sizes = [cc.cccl_get_result(w, stream)[0] for w in ws[:R]]
    red_bytes, red_status = cc.cccl_get_result(ws[R], stream)
    _, dec_status = cc.cccl_get_result(ws[R + 1], stream)
    if red_status or dec_status or 0 in sizes:
        raise RuntimeError("device status %d/%d during the first step" % (red_status, dec_status))
    check = check_against_oracle(xs_host, streams, sizes, y, n)

    warmup = max(args.warmup, 3)
    for _ in range(warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    y_plain = y.clone()

    # The timed step is one CUDA graph: the same four library calls captured
    # once (each call's workspace clear and kernel become graph nodes) and
    # replayed every step.
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step(s=side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step(s=torch.cuda.current_stream(device))
    y.zero_()
    for _ in range(warmup):
        flush.fill_(1)
        graph.replay()
    torch.cuda.synchronize()
    graph_ok = bool(torch.equal(y, y_plain))
    del y_plain

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # timed region: K graph replays, the L2 flushed before each (untimed)
    t_wall0 = time.time()
    evg = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        evg[k][0].record(stream)
        graph.replay()
        evg[k][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in evg]
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(sum(step_ms), world, device)
    # the ops one by one: K more steps of plain launches with an event pair
    # around every call (the call's workspace clear included), same flush
    op_ms = [[] for _ in range(R + 2)]
    plain_ms = []
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R + 2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        step(evs[k])
    torch.cuda.synchronize()
    t_wall1 = time.time()
    for k in range(args.steps):
        e = evs[k]
        for i in range(R + 2):
            op_ms[i].append(e[i][0].elapsed_time(e[i][1]))
        plain_ms.append(e[0][0].elapsed_time(e[R + 1][1]))

    # end to end through the same calls: pinned host inputs in, decoded result
    # out, every step.  Pipelined over three streams with two device buffer
    # sets: the upload of step k+1 and the download of step k-1 run while
    # step k computes; the timed region spans the first upload to the last
    # download.
    e2e_steps = max(2, min(args.steps, 400))
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    xs2 = [xs, [torch.empty_like(x) for x in xs]]
    ys2 = [y, torch.empty_like(y)]
    y_hosts = [y_host, torch.empty(n, dtype=torch.int16).pin_memory()]
    outs2 = [streams, [torch.empty_like(t) for t in streams]]
    reds2 = [red, torch.empty_like(red)]
    wss2 = [ws, [torch.empty_like(w) for w in ws]]
    ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_out = [torch.cuda.Event() for _ in range(e2e_steps)]

    def e2e_step(k):
        b = k % 2
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(ev_done[k - 2])  # step k-2 has finished reading this buffer set
            for r in range(R):
                xs2[b][r].copy_(pinned[r], non_blocking=True)
            ev_in[k].record(up)
        stream.wait_event(ev_in[k])
        if k >= 2:
            stream.wait_event(ev_out[k - 2])  # the result buffer of step k-2 was read out
        for r in range(R):
            cc.cccl_compress(xs2[b][r], outs2[b][r], wss2[b][r], stream)
        cc.cccl_reduce_compressed(outs2[b], n, reds2[b], wss2[b][R], stream=stream)
        cc.cccl_decompress(reds2[b], ys2[b], wss2[b][R + 1], stream=stream)
        ev_done[k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[k])
            y_hosts[b].copy_(ys2[b], non_blocking=True)
            ev_out[k].record(down)

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    for k in range(e2e_steps):
        e2e_step(k)
    down.wait_event(ev_out[e2e_steps - 1])
    e1.record(down)
    e1.synchronize()
    e2e_total = max_over_ranks(e0.elapsed_time(e1), world, device)
    last = (e2e_steps - 1) % 2
    e2e_ok = bool(torch.equal(y_hosts[last], ys2[last].cpu()))
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    bytes_step = R * 2 * n
    value = world * bytes_step * args.steps / (total_ms * 1e-3) / 1e9
    e2e_value = world * bytes_step * e2e_steps / (e2e_total * 1e-3) / 1e9

    peak, peak_kind = measured_peaks()
    mean = lambda v: sum(v) / len(v)
    ops = {}
    total_in = sum(sizes)
    algo = {"compress": 2 * n + mean(sizes), "reduce": total_in + red_bytes, "decompress": red_bytes + 2 * n}
    comp_ms = mean([mean(op_ms[r]) for r in range(R)])
    ops["compress"] = {"ms": comp_ms, "launches_per_step": R}
    ops["reduce"] = {"ms": mean(op_ms[R]), "launches_per_step": 1}
    ops["decompress"] = {"ms": mean(op_ms[R + 1]), "launches_per_step": 1}
    for name, o in ops.items():
        o["ms"] = round(o["ms"], 5)
        o["uncompressed_gbs"] = round((R if name == "reduce" else 1) * 2 * n / (o["ms"] * 1e-3) / 1e9, 1)
        o["algorithmic_bytes"] = int(algo[name])
        o["hbm_gbs"] = round(algo[name] / (o["ms"] * 1e-3) / 1e9, 1)
        o["frac_of_measured_copy"] = round(o["hbm_gbs"] / peak, 4)
        o["frac_of_8tbs_nominal"] = round(o["hbm_gbs"] / 8000.0, 4)
    dominant = max(ops, key=lambda k: ops[k]["ms"] * ops[k]["launches_per_step"])
    kname = {"compress": "compress_kernel", "reduce": "reduce_kernel", "decompress": "decompress_kernel"}[dominant]
    traffic = recorded_traffic(kname)
    roofline = {"bound": "hbm", "kernel": kname, "achieved": ops[dominant]["hbm_gbs"], "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": ops[dominant]["frac_of_measured_copy"],
                "traffic": None if traffic is None else traffic["bytes_per_launch_scaled"],
                "algorithmic_bytes_per_launch": ops[dominant]["algorithmic_bytes"]}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8+f32", "data": "synthetic",
        "config": dict(workload_config(), input_sha256=[hashlib.sha256(x.tobytes()).hexdigest()[:16]
                                                        for x in xs_host]),
        "ratio": {"compress": round(mean(sizes) / (2 * n), 5), "reduce_out": round(red_bytes / (2 * n), 5)},
        "launch": {"step": "one CUDA graph replay per step (the 4 library calls, each a workspace clear and a "
                           "kernel)", "graph_result_matches_plain": graph_ok,
                   "ops": "timed in a second pass of %d plain-launch steps, one event pair around each call "
                          "(its workspace clear included)" % args.steps,
                   "ms_per_step_plain": round(sum(plain_ms) / len(plain_ms), 5)},
        "ops": ops, "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": R * 2 * n,
                "d2h_bytes_per_step": 2 * n, "steps": e2e_steps,
                "pipelined": "uploads on one stream, steps on another, downloads on a third; step k+1's "
                             "upload and step k-1's download overlap step k (two device buffer sets)",
                "l2": "not flushed: every step uploads R x 64 MiB of input, more than the L2",
                "result_matches_device": e2e_ok},
        "gpu_launches": (R + 2) * args.steps,
        "clocks": clocks, "check": check,
        "extras": measure_extras(cc, torch, np, xs, streams, sizes, n, flush, peak) if not args.no_extras else None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(xs_host)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(xs_host)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def check_against_oracle(xs_host, streams, sizes, y, n, chunks: int = 64) -> dict:
    """Byte-exact check of sampled chunks against the oracle (not timed)."""
    import numpy as np

    import oracle

    oracle.build()
    import struct

    ok = True
    for x, s, nb in zip(xs_host, streams, sizes):
        head = s[:min(nb, 64 + 8 * (chunks + 1))].cpu().numpy().tobytes()
        offs = struct.unpack_from("<%dQ" % (chunks + 1), head, 64)
        body = s[offs[0]:offs[chunks]].cpu().numpy().tobytes()
        ref = b"".join(oracle.encode_chunk(x[c * 4096:(c + 1) * 4096]) for c in range(chunks))
        ok = ok and body == ref
    want = oracle.sum_ranks([x[:chunks * 4096] for x in xs_host])
    got = y[:chunks * 4096].cpu().numpy().view(np.uint16)
    ok = ok and bool(np.array_equal(want, got))
    return {"bit_exact_sample": ok, "sample": "first %d chunks of every stream and of the decoded sum" % chunks}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the rows timed outside the step")
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)
    return 0


if __name__ == "__main__":
    sys.exit(main())

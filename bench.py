"""Benchmark of the compressed data-parallel reduce step on GB300.

One step = the fused reduce step of a compressed allreduce over R = 8
simulated data-parallel ranks held in this GPU's memory, each rank a 256 MiB
bf16 buffer (134,217,728 values ~ N(0, 0.02), per-rank seeds) held
pre-compressed: one call of cccl_reduce_compressed, which decodes every rank's
chunks, adds them in binary32 in rank order 0..7, rounds once to bf16 and
compresses the result (decompress -> reduce -> compress in one kernel).
`value` = uncompressed gradient bytes entering the step (R * 2n) / step time,
timed on the device with CUDA events around each call, the L2 flushed (256 MiB
write, untimed) before every step, max over ranks.  The inputs (1.76 GB of
streams) are far larger than the L2 as well.  The end-to-end leg runs the same
call with the compressed streams uploaded from pinned host memory and the
result downloaded every step.  N GPUs under torchrun run N independent
replicas (weak scaling); nothing crosses GPUs.  The other workloads and
kernels (compress, decompress, the 64 MiB two-rank step, the worst case, the
KV-cache payload, fp16/fp32, ...) are timed under `extras`.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compress / decompress / fused-reduce uncompressed GB/s and % of HBM roofline; ratio"
WORKLOAD = 3          # 8 ranks x 256 MiB, N(0, 0.02), fused reduce R=8
RANKS_PER_GPU = 8     # simulated data-parallel ranks reduced on each GPU
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
E2E_MIN_STEPS = 50
E2E_WARMUP = 3
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


def workload_config(input_sha256: list[str]) -> dict:
    return {"workload": "fused decompress -> binary32 reduce in rank order -> bf16 -> compress over R=%d simulated "
                        "data-parallel ranks per GPU, each a 256 MiB bf16 buffer (134,217,728 values ~ N(0, 0.02), "
                        "per-rank seeds) held pre-compressed in HBM" % RANKS_PER_GPU,
            "n_elems": 134217728, "ranks_per_gpu": RANKS_PER_GPU, "chunk_elems": 4096,
            "l2": "flushed before every timed step (256 MiB write, untimed); the 1.76 GB of input streams are far "
                  "larger than the L2 as well",
            "parallelism": "replicas (weak scaling, no cross-GPU traffic)",
            "input_sha256": input_sha256}


def input_hashes(xs_host) -> list[str]:
    return [hashlib.sha256(x.tobytes()).hexdigest()[:16] for x in xs_host]


# ---------------------------------------------------------------- clocks
# NVML (read-only queries) through ctypes, every millisecond; nvidia-smi at
# 100 ms when NVML cannot be loaded.  Clock event reason bits of NVML.
_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _NvmlSource:
    def __init__(self, torch_index: int):
        import torch

        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self.lib.nvmlInit_v2.restype = ctypes.c_int
        rc = self.lib.nvmlInit_v2()
        if rc != 0:
            raise OSError("nvmlInit_v2 returned %d" % rc)
        self.handle = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(torch_index)
        rc = -1
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            text = str(uuid)
            if not text.startswith("GPU-"):
                text = "GPU-" + text
            rc = self.lib.nvmlDeviceGetHandleByUUID(text.encode(), ctypes.byref(self.handle))
        if rc != 0 and hasattr(props, "pci_bus_id"):
            bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                        getattr(props, "pci_device_id", 0))
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle))
        if rc != 0:
            raise OSError("no NVML handle for torch device %d (rc %d)" % (torch_index, rc))
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        mhz, mx, mw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz))       # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))
        self.reasons_fn(self.handle, ctypes.byref(reasons))
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw))
        return float(mhz.value), float(mx.value), int(reasons.value), mw.value / 1000.0


class ClockSampler:
    """SM clock, its maximum, clock event reasons and power while the work runs."""

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, torch_index: int, period_s: float = 0.001):
        self.samples: list[tuple[float, float, float, set, float]] = []
        self.period = period_s
        self.source = None
        self.note = None
        self.stop_flag = threading.Event()
        self.thread = None
        self.proc = None
        try:
            self.nvml = _NvmlSource(torch_index)
            self.source = "nvml"
        except Exception as e:  # no driver, no device, no NVML: fall back, and say why
            self.nvml = None
            self.note = "NVML unavailable (%s); nvidia-smi at 100 ms" % e
            self.smi_index = torch_index

    def start(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.smi_index), "--query-gpu=" + self.SMI_FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                text=True)
            self.source = "nvidia-smi"
        except OSError as e:
            self.note = (self.note or "") + "; nvidia-smi could not start: %s" % e
            return
        self.thread = threading.Thread(target=self._smi_loop, daemon=True)
        self.thread.start()

    def _nvml_loop(self):
        while not self.stop_flag.is_set():
            mhz, mx, bits, w = self.nvml.sample()
            self.samples.append((time.time(), mhz, mx, {n for b, n in _REASON_BITS.items() if bits & b}, w))
            time.sleep(self.period)

    def _smi_loop(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                reasons = {n for n, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                              "sw_power_cap"), parts[3:7]) if v.lower().startswith("active")}
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), reasons, float(parts[2])))
            except ValueError:
                continue

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                _, err = self.proc.communicate(timeout=5)
                if self.proc.returncode not in (0, -15, None) and err:
                    self.note = (self.note or "") + "; nvidia-smi rc %s: %s" % (self.proc.returncode, err.strip()[:200])
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        sel = [s for s in self.samples if t0 <= s[0] <= t1]
        reasons = sorted(set().union(*[s[3] for s in sel])) if sel else []
        out = {"sm_mhz": statistics.median([s[1] for s in sel]) if sel else None,
               "sm_max_mhz": max(s[2] for s in sel) if sel else None,
               "reasons": reasons, "samples": len(sel),
               "power_w_max": round(max(s[4] for s in sel), 1) if sel else None,
               "source": self.source, "window_s": round(t1 - t0, 3)}
        if self.note:
            out["note"] = self.note
        return out


# ---------------------------------------------------------------- the oracle as a CPU baseline
def oracle_reduce_seconds(xs, start_chunk: int, chunks: int) -> tuple[float, int]:
    """The oracle doing the step on chunks [start_chunk, start_chunk + chunks)
    of every rank: the ranks' pieces compressed first (the step's inputs are
    held pre-compressed; not timed), then the fused reduce, timed."""
    import oracle

    a = start_chunk * 4096
    b = min(xs[0].size, a + chunks * 4096)
    streams = [oracle.compress(x[a:b]) for x in xs]
    t = time.perf_counter()
    oracle.reduce(streams, b - a)
    return time.perf_counter() - t, b - a


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


def cpu_baseline(xs, budget_s: float = 12.0) -> dict:
    """The oracle, as it stands, single-threaded, on windows of 256 chunks
    spread over the whole workload, until about budget_s of reduce time."""
    import oracle

    oracle.build()
    n_chunks = xs[0].size // 4096
    window = 256
    total_t, total_n, k = 0.0, 0, 0
    while total_t < budget_s and k < 512:
        start = (k * 7919 * window) % max(1, n_chunks - window)
        dt, n = oracle_reduce_seconds(xs, start, window)
        total_t += dt
        total_n += n
        k += 1
    gbs = len(xs) * 2 * total_n / total_t / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
            "sample": "the step (fused reduce of %d pre-compressed ranks) on %d windows of %d chunks spread over the "
                      "workload (%d values per rank), %.1f s of reduce time, single-threaded C oracle; the "
                      "windows' compression is not timed" % (len(xs), k, window, total_n, total_t)}


def cpu_baseline_all_cores(xs, budget_s: float = 8.0) -> dict:
    """The oracle, as it stands, on every host core at once: each thread
    reduces its own windows of chunks (the oracle is single-threaded C; the
    threads share nothing)."""
    import concurrent.futures as cf

    import oracle

    oracle.build()
    cores = max(1, os.cpu_count() or 1)
    n_chunks = xs[0].size // 4096
    window = 128
    per = max(window, n_chunks // cores)

    def one(i, rnd):
        start = (i * per + rnd * window) % max(1, n_chunks - window)
        return oracle_reduce_seconds(xs, start, window)

    total_n, busy, rounds = 0, 0.0, 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(cores) as ex:
        while time.perf_counter() - t0 < budget_s and rounds < 16:
            res = list(ex.map(lambda i: one(i, rounds), range(cores)))
            total_n += sum(n for _, n in res)
            busy += max(t for t, _ in res)
            rounds += 1
    gbs = len(xs) * 2 * total_n / busy / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu": cpu_model(),
            "sample": "%d threads, each the step on its own %d-chunk windows, %d round(s); time = the slowest thread's "
                      "reduce time per round, summed (%.1f s); compression of the windows not timed"
                      % (cores, window, rounds, busy)}


def run_reference(args, rank: int, world: int) -> None:
    """The reference arm: the CPU oracle, as it stands, on this host's cores,
    doing the same step (the fused reduce of the 8 pre-compressed ranks) on a
    bounded sample of chunks per step, rotating through the workload."""
    import oracle
    import workloads

    oracle.build()
    workloads.build()
    if rank != 0:
        return
    xs = [workloads.generate(WORKLOAD, r) for r in simulated_ranks(0)]
    n_chunks = xs[0].size // 4096
    steps, warmup = args.steps, max(args.warmup, 3)
    # each step: a window of chunks sized so that the whole run takes about
    # two minutes of reduce time
    per_step_s = 100.0 / (steps + warmup)
    probe_t, _ = oracle_reduce_seconds(xs, 0, 16)
    chunks = max(1, min(n_chunks, int(per_step_s / (probe_t / 16))))
    offs = 0
    total_t, total_n = 0.0, 0
    for i in range(warmup + steps):
        start = offs % max(1, n_chunks - chunks)
        dt, n = oracle_reduce_seconds(xs, start, chunks)
        offs += chunks
        if i >= warmup:
            total_t += dt
            total_n += n
    value = RANKS_PER_GPU * 2 * total_n / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(1e3 * total_t / steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8+f32",
        "data": "synthetic", "config": workload_config(input_hashes(xs)),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
                         "sample": "%d chunks of every rank per step, rotating through the workload; the chunks' "
                                   "compression is not timed (the step's inputs are held pre-compressed)" % chunks},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- rows beyond the step
KV_BLOCK = 16 * 8 * 128  # 16 tokens x 8 heads x 128 dim


def make_timer(torch, flush, stream, reps: int):
    """Median CUDA-event time (ms) of fn() on `stream`, the L2 flushed before
    every repetition (untimed), after 3 untimed repetitions."""
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
    return timed


def op_row(ms, algo, uncompressed, peak, **kw):
    d = {"ms": round(ms, 5), "algorithmic_bytes": int(algo),
         "uncompressed_gbs": round(uncompressed / (ms * 1e-3) / 1e9, 1),
         "hbm_gbs": round(algo / (ms * 1e-3) / 1e9, 1),
         "frac_of_measured_copy": round(algo / (ms * 1e-3) / 1e9 / peak, 4),
         "frac_of_8tbs_nominal": round(algo / (ms * 1e-3) / 1e9 / 8000.0, 4)}
    d.update(kw)
    return d


def measure_extras(cc, torch, np, timed, stream, peak, x0, red, red_bytes, n3) -> dict:
    """The kernels and workloads outside the timed step, each op timed alone."""
    import workloads

    out = {}
    tab3 = 8 * (-(-n3 // 4096))
    # the step's other kernels on its own data: compress of rank 0's buffer,
    # decompress of the reduced stream (the receiver's decode)
    s0 = cc.empty_stream(n3)
    ws = cc.empty_workspace(n3)
    ms_c = timed(lambda: cc.cccl_compress(x0, s0, ws, stream=stream))
    b0, st_c = cc.cccl_get_result(ws, stream)
    out["workload3_compress"] = op_row(ms_c, 2 * n3 + b0 + tab3, 2 * n3, peak, status=st_c,
                                       ratio=round(b0 / (2 * n3), 5),
                                       workload="rank 0's 256 MiB buffer of the timed step")
    y = torch.empty(n3, dtype=torch.int16, device=x0.device)
    ms_d = timed(lambda: cc.cccl_decompress(red[:red_bytes], y, ws, stream=stream))
    _, st_d = cc.cccl_get_result(ws, stream)
    out["workload3_decompress_reduced"] = op_row(ms_d, red_bytes + tab3 + 2 * n3, 2 * n3, peak, status=st_d,
                                                 workload="the step's reduced stream, decoded")
    del s0, y
    # the 64 MiB gradient-like buffer on two ranks: compress each, fused
    # reduce, decompress the result
    n = workloads.SIZES[2]
    tab = 8 * (-(-n // 4096))
    xs = [torch.from_numpy(workloads.generate(2, r).view(np.int16)).to(x0.device) for r in range(2)]
    ss = [cc.empty_stream(n) for _ in xs]
    ws2 = cc.empty_workspace(n)
    sizes = []
    for x, s_ in zip(xs, ss):
        cc.cccl_compress(x, s_, ws2, stream=stream)
        sizes.append(cc.cccl_get_result(ws2, stream)[0])
    ms_c2 = timed(lambda: cc.cccl_compress(xs[0], ss[0], ws2, stream=stream))
    red2 = cc.empty_stream(n)
    ins = [s_[:b] for s_, b in zip(ss, sizes)]
    ms_r2 = timed(lambda: cc.cccl_reduce_compressed(ins, n, red2, ws2, stream=stream))
    rb2, st_r2 = cc.cccl_get_result(ws2, stream)
    y2 = torch.empty(n, dtype=torch.int16, device=x0.device)
    ms_d2 = timed(lambda: cc.cccl_decompress(red2[:rb2], y2, ws2, stream=stream))
    step = 2 * ms_c2 + ms_r2 + ms_d2
    w2 = "gradient-like 64 MiB bf16 buffer (33,554,432 values ~ N(0, 1e-3), 1% of positions x100)"
    out["workload2_compress"] = op_row(ms_c2, 2 * n + sizes[0] + tab, 2 * n, peak,
                                       ratio=round(sizes[0] / (2 * n), 5), workload=w2)
    out["workload2_reduce_r2"] = op_row(ms_r2, sum(sizes) + 2 * tab + rb2 + tab, 4 * n, peak, status=st_r2,
                                        workload=w2 + ", 2 ranks")
    out["workload2_decompress"] = op_row(ms_d2, rb2 + tab + 2 * n, 2 * n, peak, workload=w2 + ", reduced stream")
    out["workload2_step"] = {"ms": round(step, 5), "uncompressed_gbs": round(4 * n / (step * 1e-3) / 1e9, 1),
                             "workload": w2 + ": compress both ranks, fused reduce R=2, decompress (sum of the ops "
                                          "timed alone)"}
    # local rank-0 buffer + one compressed remote rank (selective compression)
    ms = timed(lambda: cc.cccl_reduce_mixed(xs[0], [ins[1]], red2, ws2, stream=stream))
    out_bytes, st = cc.cccl_get_result(ws2, stream)
    out["reduce_mixed"] = op_row(ms, 2 * n + sizes[1] + out_bytes, 4 * n, peak, status=st,
                                 workload="local rank-0 buffer (uncompressed) + 1 compressed remote rank of " + w2)
    # KV-cache blocks of the [32, 2, 4096, 8, 128] shape: 4096 of a pool of 8192 blocks, shuffled
    n_pool, n_blk = 8192, 4096
    pool = torch.from_numpy(workloads.generate(4, 0, count=n_pool * KV_BLOCK).view(np.int16)).to(x0.device)
    table = torch.from_numpy(np.random.default_rng(7).permutation(n_pool)[:n_blk].astype(np.int32)).to(x0.device)
    npg = n_blk * KV_BLOCK
    s_pg = cc.empty_stream(npg)
    ws_pg = cc.empty_workspace(npg)
    ms_c = timed(lambda: cc.cccl_compress_paged(pool, KV_BLOCK, table, s_pg, ws_pg, stream=stream))
    pbytes, st_c = cc.cccl_get_result(ws_pg, stream)
    target = torch.empty_like(pool)
    ms_d = timed(lambda: cc.cccl_decompress_paged(s_pg[:pbytes], target, KV_BLOCK, table, ws_pg, stream=stream))
    _, st_d = cc.cccl_get_result(ws_pg, stream)
    ok = bool(torch.equal(target.view(n_pool, KV_BLOCK)[table.long()], pool.view(n_pool, KV_BLOCK)[table.long()]))
    kv = ("4096 KV-cache blocks of 16 tokens x 8 heads x 128 dim (64 Mi values) gathered through a shuffled block "
          "table from a pool of 8192")
    out["compress_paged"] = op_row(ms_c, 2 * npg + pbytes, 2 * npg, peak, status=st_c, workload=kv,
                                   ratio=round(pbytes / (2 * npg), 5))
    out["decompress_paged"] = op_row(ms_d, 2 * npg + pbytes, 2 * npg, peak, status=st_d, workload=kv,
                                     round_trip_exact=ok)
    del pool, target, s_pg
    # window-base variant (stream version 2) next to the minimum-base stream
    for name, x in (("compress_window", xs[0]),
                    ("compress_window_specials",
                     torch.from_numpy(workloads.generate(5, 0, start=1 << 27, count=n).view(np.int16)).to(x0.device))):
        s_w = cc.empty_stream(n)
        ms_w = timed(lambda: cc.cccl_compress_window(x, s_w, ws2, stream=stream))
        wbytes, st_w = cc.cccl_get_result(ws2, stream)
        cc.cccl_compress(x, s_w, ws2, stream=stream)
        v1bytes, _ = cc.cccl_get_result(ws2, stream)
        out[name] = op_row(ms_w, 2 * n + wbytes, 2 * n, peak, status=st_w,
                           workload=w2 if name == "compress_window" else
                           "64 MiB of N(0, 1) with 0.1% each NaN, +-Inf, +-0, subnormals (second half of the worst-case "
                           "buffer)", ratio=round(wbytes / (2 * n), 5), ratio_min_base=round(v1bytes / (2 * n), 5))
    del xs, ss, red2, y2
    torch.cuda.empty_cache()
    out.update(measure_dtypes(cc, torch, np, n, timed, stream, peak))
    out.update(measure_workloads(cc, torch, np, timed, stream, peak))
    return out


def measure_workloads(cc, torch, np, timed, stream, peak) -> dict:
    """The 512 MiB workloads at their full sizes, each op timed alone: the
    KV-cache tensor round trip; the worst case (half incompressible) round
    trip and its R=4 fused reduce.  Inputs are far larger than the L2."""
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
        xs = [torch.from_numpy(workloads.generate_typed(dtype, 2, r).view(np.int16 if item == 2 else np.int32))
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
    stream = torch.cuda.current_stream(device)
    cap = cc.cccl_compress_bound(n)
    tab = 8 * (-(-n // 4096))
    # the ranks' buffers, held pre-compressed in HBM (compression not timed)
    streams, sizes = [], []
    ws_c = cc.empty_workspace(n)
    x0 = None
    for r, xh in enumerate(xs_host):
        x = torch.from_numpy(xh.view(np.int16)).to(device)
        s_ = torch.empty(cap, dtype=torch.uint8, device=device)
        cc.cccl_compress(x, s_, ws_c, stream=stream)
        b, st = cc.cccl_get_result(ws_c, stream)
        if st != 0:
            raise RuntimeError("compress of rank %d: device status %d" % (r, st))
        streams.append(s_)
        sizes.append(b)
        if r == 0:
            x0 = x
        else:
            del x
    ins = [s_[:b] for s_, b in zip(streams, sizes)]
    red = torch.empty(cap, dtype=torch.uint8, device=device)
    ws = cc.empty_workspace(n)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def step(s=stream):
        cc.cccl_reduce_compressed(ins, n, red, ws, stream=s)

    # one untimed step: size, status and a sampled check against the oracle
    step()
    red_bytes, red_status = cc.cccl_get_result(ws, stream)
    if red_status:
        raise RuntimeError("device status %d during the first step" % red_status)
    check = check_against_oracle(xs_host, streams, sizes, red, red_bytes, n)

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    warmup = max(args.warmup, 3)
    for _ in range(warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # timed region: K steps, each one C-ABI call (workspace clear + kernel),
    # an event pair around it; the L2 flushed before each (untimed)
    t_wall0 = time.time()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(sum(step_ms), world, device)
    same_result = cc.cccl_get_result(ws, stream) == (red_bytes, 0)

    # end to end through the same call: the compressed streams uploaded from
    # pinned host memory and the result stream (its full bound, which holds
    # the stream's own size) downloaded every step.  Pipelined over three
    # streams with two device buffer sets: the upload of step k+1 and the
    # download of step k-1 run while step k computes.  Untimed warm-up steps
    # cover both buffer sets first.
    e2e_steps = max(E2E_MIN_STEPS, args.steps)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    pinned_in = [torch.empty(b, dtype=torch.uint8).pin_memory() for b in sizes]
    for p, s_, b in zip(pinned_in, streams, sizes):
        p.copy_(s_[:b])
    dev_in = [[torch.empty(b, dtype=torch.uint8, device=device) for b in sizes] for _ in range(2)]
    dev_out = [red, torch.empty_like(red)]
    dev_ws = [ws, torch.empty_like(ws)]
    host_out = [torch.empty(cap, dtype=torch.uint8).pin_memory() for _ in range(2)]
    n_total = E2E_WARMUP + e2e_steps
    ev_in = [torch.cuda.Event() for _ in range(n_total)]
    ev_done = [torch.cuda.Event() for _ in range(n_total)]
    ev_out = [torch.cuda.Event() for _ in range(n_total)]

    def e2e_step(k):
        b = k % 2
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(ev_done[k - 2])  # step k-2 has finished reading this buffer set
            for d, p in zip(dev_in[b], pinned_in):
                d.copy_(p, non_blocking=True)
            ev_in[k].record(up)
        stream.wait_event(ev_in[k])
        if k >= 2:
            stream.wait_event(ev_out[k - 2])  # the result buffer of step k-2 was read out
        cc.cccl_reduce_compressed(dev_in[b], n, dev_out[b], dev_ws[b], stream=stream)
        ev_done[k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[k])
            host_out[b].copy_(dev_out[b], non_blocking=True)
            ev_out[k].record(down)

    for k in range(E2E_WARMUP):
        e2e_step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    for k in range(E2E_WARMUP, n_total):
        e2e_step(k)
    down.wait_event(ev_out[n_total - 1])
    e1.record(down)
    e1.synchronize()
    t_wall2 = time.time()
    e2e_total = max_over_ranks(e0.elapsed_time(e1), world, device)
    last = (n_total - 1) % 2
    e2e_ok = bool(torch.equal(host_out[last][:red_bytes], red[:red_bytes].cpu()))
    del dev_in, pinned_in, host_out
    torch.cuda.empty_cache()

    bytes_step = R * 2 * n
    value = world * bytes_step * args.steps / (total_ms * 1e-3) / 1e9
    e2e_value = world * bytes_step * e2e_steps / (e2e_total * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    ms_mean = sum(step_ms) / len(step_ms)
    algo = sum(sizes) + R * tab + red_bytes + tab
    ops = {"reduce": op_row(ms_mean, algo, bytes_step, peak, launches_per_step=1,
                            ms_median=round(statistics.median(step_ms), 5), ms_min=round(min(step_ms), 5))}
    traffic = recorded_traffic("reduce_kernel")
    roofline = {"bound": "hbm", "kernel": "reduce_kernel", "achieved": ops["reduce"]["hbm_gbs"], "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": ops["reduce"]["frac_of_measured_copy"],
                "frac_of_8tbs_nominal": ops["reduce"]["frac_of_8tbs_nominal"],
                "traffic": None if traffic is None else traffic["bytes_per_launch_scaled"],
                "algorithmic_bytes_per_launch": int(algo),
                "duration": "mean CUDA-event time of the timed calls (each call: the workspace clear and the kernel)"}
    extras = None
    if not args.no_extras:
        timed = make_timer(torch, flush, stream, reps=20)
        extras = measure_extras(cc, torch, np, timed, stream, peak, x0, red, red_bytes, n)
    t_wall3 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    clocks["whole_run"] = {k: v for k, v in sampler.summary(t_wall0, t_wall3).items() if k != "note"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8+f32", "data": "synthetic",
        "config": workload_config(input_hashes(xs_host)),
        "ratio": {"inputs": round(sum(sizes) / (R * 2 * n), 5), "reduce_out": round(red_bytes / (2 * n), 5)},
        "launch": {"step": "one cccl_reduce_compressed call per step (a workspace clear and one kernel)",
                   "result_unchanged_after_timing": same_result},
        "ops": ops, "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": int(sum(sizes)),
                "d2h_bytes_per_step": int(cap), "steps": e2e_steps, "warmup_steps": E2E_WARMUP,
                "pipelined": "uploads on one stream, steps on another, downloads on a third; step k+1's "
                             "upload and step k-1's download overlap step k (two device buffer sets)",
                "result_matches_device": e2e_ok},
        "gpu_launches": args.steps,
        "clocks": clocks, "check": check,
        "extras": extras,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(xs_host)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(xs_host)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def check_against_oracle(xs_host, streams, sizes, red, red_bytes, n, chunks: int = 16) -> dict:
    """Byte-exact check against the oracle, not timed: three windows of
    `chunks` chunks (start, middle, end) of every rank's stream and of the
    reduced stream."""
    import struct

    import numpy as np

    import oracle

    oracle.build()
    n_chunks = -(-n // 4096)
    ok = True
    windows = [0, n_chunks // 2, n_chunks - chunks]

    def chunk_bytes(s, nbytes, c0):
        offs = struct.unpack_from("<%dQ" % (chunks + 1), s[64 + 8 * c0:64 + 8 * (c0 + chunks + 1)].cpu().numpy()
                                  .tobytes()) if c0 + chunks < n_chunks else None
        if offs is None:
            first = struct.unpack_from("<Q", s[64 + 8 * c0:64 + 8 * c0 + 8].cpu().numpy().tobytes())[0]
            return s[first:nbytes].cpu().numpy().tobytes()
        return s[offs[0]:offs[chunks]].cpu().numpy().tobytes()

    for c0 in windows:
        a, b = c0 * 4096, min(n, (c0 + chunks) * 4096)
        for x, s, nb in zip(xs_host, streams, sizes):
            ref = b"".join(oracle.encode_chunk(x[c * 4096:(c + 1) * 4096]) for c in range(c0, c0 + chunks))
            ok = ok and chunk_bytes(s, nb, c0) == ref
        part = [oracle.compress(x[a:b]) for x in xs_host]
        want = oracle.reduce(part, b - a)
        body = want[oracle.data_start(b - a):].tobytes()
        ok = ok and chunk_bytes(red, red_bytes, c0) == body
    return {"bit_exact_sample": bool(ok),
            "sample": "chunks [c, c+%d) for c in %s of every rank's stream and of the reduced stream" % (chunks, windows)}


def run_case(args) -> None:
    """One kernel alone, for a profiler: --case OP,WORKLOAD,RANKS,VALUES with OP
    compress, decompress or reduce.  The inputs (VALUES values of WORKLOAD's
    recipe per rank) are generated and, for decompress and reduce, compressed
    first; then the op runs --warmup + --steps times, one call after another
    on the current stream, and one JSON line gives its mean CUDA-event time."""
    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import compression_coupled_collectives_gb300 as cc
    import workloads

    op, w, ranks, n = args.case.split(",")
    w, ranks, n = int(w), int(ranks), int(n)
    stream = torch.cuda.current_stream()
    xs = [torch.from_numpy(workloads.generate(w, r, count=n, n=max(n, workloads.SIZES[w])).view(np.int16)).cuda()
          for r in range(ranks)]
    ws = cc.empty_workspace(n)
    streams = []
    for x in xs:
        s_ = cc.empty_stream(n)
        cc.cccl_compress(x, s_, ws, stream=stream)
        streams.append(s_[:cc.cccl_get_result(ws, stream)[0]])
    out = cc.empty_stream(n)
    y = torch.empty(n, dtype=torch.int16, device="cuda")
    calls = {"compress": lambda: cc.cccl_compress(xs[0], out, ws, stream=stream),
             "decompress": lambda: cc.cccl_decompress(streams[0], y, ws, stream=stream),
             "reduce": lambda: cc.cccl_reduce_compressed(streams, n, out, ws, stream=stream)}
    call = calls[op]
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    e1.synchronize()
    _, st = cc.cccl_get_result(ws, stream)
    print(json.dumps({"case": args.case, "ms_mean": round(e0.elapsed_time(e1) / args.steps, 5), "status": st,
                      "input_bytes": [int(t.numel() * t.element_size()) for t in (streams if op != "compress" else [xs[0]])]}))
    if st != 0:
        raise RuntimeError("device status %d" % st)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the rows timed outside the step")
    ap.add_argument("--case", help="OP,WORKLOAD,RANKS,VALUES: time one kernel alone (for profilers)")
    args = ap.parse_args(argv)
    if args.case:
        run_case(args)
        return 0
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)
    return 0


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python3
"""Benchmark of the DeepSelect top-k library on GB300.

One step = one ds_topk call over one batch of the workload (all rows): the
random block order, the streaming filter, the in-loop radix selects, the
split-row merge and the final sort.  The headline workload is the largest
one that fits a GPU, the sampling-logit batch (256 rows x 128000 bf16,
k = 50, B = B2 = 1024); the other workloads are reported under "per_config",
each with the CPU oracle timed on a bounded sample of its rows.

Timing: inputs are resident in HBM, rotated over enough replicas that the
replicas together are at least four times the L2 size, so every step reads
its batch from DRAM.  The K timed launches are replayed from CUDA graphs and
bracketed by CUDA events on the launching stream (plus a barrier and a
device synchronize on both sides).  "e2e" times the host-buffer entry
points: pinned host input -> device -> top-k -> pinned host output every
step, four steps in flight on four streams (ds_topk_host_async), and also
synchronised every step (ds_topk_host).

Multi-GPU (torchrun): rows are independent, so the batch is partitioned into
contiguous row ranges (row_range), one per rank; every rank selects its own
rows and writes its own slice of the outputs, with no data exchange.  By
default (--scaling weak) the batch holds `rows` rows per rank; with
--scaling strong the workload's rows are split across the ranks.  Rank 0
prints the total rows of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (single thread, the plain definition
by full sort) on the same workload, each step a bounded sample of rows.
"""
import argparse
import hashlib
import json
import math
import os
import platform
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "top-k rows/s and input-read HBM GB/s (fraction of GB300 peak) per config"
UNIT = "rows/s"
MAIN = "sampling_logits_bf16"
LONG_ROW_NAME = "long_row_fp32"
SEED = 0x5EED5EED
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = [os.path.join(ROOT, "top_selection_deepselect_gb300", "csrc", f)
                  for f in ("ds_topk.cu", "ds_device.cuh", "ds_kernel.cuh", "ds_stream.cuh",
                            "ds_kernels_fp32.cu", "ds_kernels_bf16.cu", "ds_kernels_fp16.cu")]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000,
                    help="timed steps (the default keeps the timed region long enough for "
                         "clock samples to fall inside it)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=MAIN, choices=workloads.CONFIG_ORDER + [LONG_ROW_NAME],
                    help="%s: one row over the whole GPU (ds_topk_long_row); the extras, the "
                         "end-to-end number and the reference arm cover the matrix workloads "
                         "only" % LONG_ROW_NAME)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip per-config lines, torch.topk and the CPU baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--e2e-steps", type=int, default=200, help="0: same as --steps")
    ap.add_argument("--burn-seconds", type=float, default=0.5,
                    help="extra untimed back-to-back warm-up before the timed region")
    ap.add_argument("--scaling", choices=["weak", "strong"], default="weak",
                    help="weak: every rank selects `rows` rows of a batch of rows x ranks; "
                         "strong: the workload's rows are split across the ranks")
    ap.add_argument("--cpu-seconds-per-config", type=float, default=3.0)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def kernel_source_hash():
    """Hash of the kernel sources' code: comments and blank space are left
    out, so a profile summary stays valid across comment-only edits."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_name(plan):
    """The kernel a call with this plan launches (calls without counters use
    the free-running kernel when their rows take 16-byte copies)."""
    return "deepselect_stream_kernel" if plan and plan.get("kernel") == 1 else "deepselect_topk_kernel"


def profile_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources."""
    path = os.path.join(PROFILE_DIR, "%s__%s.txt" % (kernel, workload))
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, _, v = line.partition(":")
                fields[k.strip()] = v.strip()
    if fields.get("source_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Clock / throttle samples taken by a background thread while the GPU
    works, every ~50 ms: read-only NVML queries in this process (ctypes on
    libnvidia-ml), or one complete nvidia-smi query per sample if NVML
    cannot be loaded."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvml.h)
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}

    def __init__(self, index):
        self.index = int(index)
        self.samples = []  # (sm_mhz, max_mhz, reason names)
        self.thread = None
        self.stop_flag = False
        self.error = None
        self.nvml = None
        self.handle = None

    def _nvml_open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            rc = lib.nvmlInit_v2()
            if rc != 0:
                self.error = "nvmlInit_v2 returned %d" % rc
                return False
            h = ctypes.c_void_p()
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h))
            if rc != 0:
                self.error = "nvmlDeviceGetHandleByIndex_v2 returned %d" % rc
                return False
            self.nvml, self.handle = lib, h
            return True
        except Exception as ex:  # no NVML here: fall back to nvidia-smi
            self.error = "nvml: %r" % (ex,)
            return False

    def _nvml_sample(self):
        import ctypes
        sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(sm)) != 0:  # NVML_CLOCK_SM
            return None
        if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) != 0:
            return None
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        reasons = set()
        if fn(self.handle, ctypes.byref(rs)) == 0:
            reasons = {n for n, b in self.REASON_BITS.items() if rs.value & b}
        return float(sm.value), float(mx.value), reasons

    def _smi_sample(self):
        # a library path that points at the toolkit's driver stubs would make
        # nvidia-smi load a stub NVML, so the child gets a clean one
        env = {k: v for k, v in os.environ.items() if k not in ("LD_LIBRARY_PATH", "LD_PRELOAD")}
        out = ""
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                "--format=csv,noheader,nounits"], capture_output=True, text=True,
                               timeout=10, env=env)
            out = r.stdout.strip()
            f = out.split(", ")
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            return (float(f[1]), float(f[2]),
                    {n for n, v in zip(names, f[5:9]) if v.strip() == "Active"})
        except Exception as ex:  # recorded, not fatal
            if "nvidia-smi" not in (self.error or ""):
                self.error = (self.error + "; " if self.error else "") + "nvidia-smi: %s" % (out[:80] or repr(ex))
            return None

    def _loop(self):
        use_nvml = self._nvml_open()
        while not self.stop_flag:
            smp = self._nvml_sample() if use_nvml else self._smi_sample()
            if smp is not None:
                self.samples.append(smp)
            time.sleep(0.05)

    def start(self):
        import threading
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 5.0:  # the sampler is running
            time.sleep(0.02)

    def stop(self):
        if self.thread is None:
            return None
        n_before = len(self.samples)
        t0 = time.perf_counter()
        while len(self.samples) == n_before and time.perf_counter() - t0 < 2.0:
            time.sleep(0.02)  # at least one sample after the timed steps were enqueued
        self.stop_flag = True
        self.thread.join(timeout=15)
        if not self.samples:
            return {"error": self.error or "no clock samples"}
        sm = [x[0] for x in self.samples]
        reasons = set()
        for x in self.samples:
            reasons |= x[2]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(x[1] for x in self.samples),
                "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvml" if self.nvml is not None else "nvidia-smi"}


def rank_rows(rank, world, rows, scaling):
    """This rank's contiguous row range [r0, r1) of the batch and the batch's
    row count: weak scaling gives every rank `rows` rows of a batch of
    rows * world, strong scaling splits `rows` (row_range of the package)."""
    import top_selection_deepselect_gb300 as ds
    total = rows * world if scaling == "weak" else rows
    r0, r1 = ds.row_range(rank, world, total)
    return r0, r1, total


def reduce_over_ranks(ms, rows, dist, device="cpu"):
    """Slowest rank's time and the rows all ranks processed (each rank selects
    its own row range; nothing but these two numbers is exchanged)."""
    if dist is None:
        return ms, rows
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    r = torch.tensor([rows], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(r, op=dist.ReduceOp.SUM)
    return float(t.item()), int(r.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def cfg_desc(c, name, plan=None):
    d = {"workload": name, "rows": c["rows"], "N": c["N"], "k": c["k"], "B": c["B"],
         "B2": c["B2"], "dtype": c["dtype"], "desc": c["desc"]}
    if plan:
        d["plan"] = plan
    return d


def data_desc(name):
    """What the synthetic rows stand in for (no public dataset is named)."""
    what = {"small_fp32": "a small score row", "dsa_index_bf16": "DSA index scores",
            "dsa_decode_ragged_fp32": "DSA long-context decode scores",
            "sampling_logits_bf16": "sampling logits",
            "adversarial_fp32": "adversarially ordered and heavily tied rows",
            LONG_ROW_NAME: "one long score row"}.get(name, name)
    return "synthetic (seeded; stands in for %s)" % what


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def oracle_rows_per_s(name, seconds=None, steps=None, warmup=0, rows_per_step=4):
    import oracle
    c = workloads.CONFIGS[name]
    bits, row_len = workloads.config_inputs(name)
    rows = c["rows"]
    step_rows = max(1, min(rows_per_step, rows))

    def one_step(i):
        r0 = (i * step_rows) % rows
        sel = [(r0 + j) % rows for j in range(step_rows)]
        rl = None if row_len is None else row_len[sel]
        oracle.topk(np.ascontiguousarray(bits[sel]), c["dtype"], c["k"], row_len=rl)

    for i in range(warmup):
        one_step(i)
    done = 0
    t0 = time.perf_counter()
    if steps is not None:
        for i in range(steps):
            one_step(warmup + i)
        done = steps
    else:
        while True:
            one_step(warmup + done)
            done += 1
            if time.perf_counter() - t0 >= seconds:
                break
    dt = time.perf_counter() - t0
    return done * step_rows / dt, dt, done, step_rows


SPEC_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (context beside the measured copy bandwidth)


def host_cpu():
    """Model name and logical core count of the host, for the CPU baseline lines."""
    model = platform.processor() or platform.machine()
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    key, val = line.split(":", 1)
                    fields.setdefault(key.strip().lower(), val.strip())
    except OSError:
        pass
    if "model name" in fields:
        model = fields["model name"]
    elif "cpu part" in fields:
        # Arm: implementer and part numbers (0x41 / 0xd4f is Neoverse V2)
        known = {("0x41", "0xd4f"): "Arm Neoverse V2"}
        key = (fields.get("cpu implementer", ""), fields["cpu part"])
        model = known.get(key, "Arm implementer %s part %s" % key)
    return {"model": model, "logical_cores": os.cpu_count()}


def run_reference(args, rank, world):
    if rank != 0:
        return
    name = args.workload
    if name == LONG_ROW_NAME:
        raise SystemExit("the reference arm times the matrix workloads; %s has none" % name)
    c = workloads.CONFIGS[name]
    rate, dt, done, step_rows = oracle_rows_per_s(name, steps=args.steps, warmup=args.warmup,
                                                  rows_per_step=1)
    sample = "%d steps x %d row of %s (rows cycled), single thread" % (done, step_rows, name)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(done, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": c["dtype"], "data": data_desc(name),
        "config": cfg_desc(c, name),
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_cpu()},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Workload:
    """Device-resident replicas of one workload plus the launch closure.
    `local_rows` = the rows [lr0, lr1) of the workload this rank selects
    (all of them unless the rows are split across ranks)."""

    def __init__(self, name, dev, torch, ds, l2_bytes, max_bytes=8 << 30, local_rows=None):
        self.name = name
        self.c = c = workloads.CONFIGS[name]
        self.torch = torch
        self.ds = ds
        bits, row_len = workloads.config_inputs(name)
        self.bits, self.row_len_np = bits, row_len
        self.esz = 4 if c["dtype"] == "fp32" else 2
        self.code = ds.DS_FP32 if c["dtype"] == "fp32" else ds.DS_BF16
        tdt = torch.float32 if c["dtype"] == "fp32" else torch.bfloat16
        host = torch.from_numpy(bits.view(np.int32 if c["dtype"] == "fp32" else np.int16))
        one = host.to(dev).view(tdt)
        nbytes = one.numel() * self.esz
        # replicas whose total is >= 4x L2, at most 512 launches per graph
        self.replicas = int(max(2, min(math.ceil(4 * l2_bytes / nbytes), max_bytes // nbytes, 512)))
        self.l2_defeated = self.replicas * nbytes >= 4 * l2_bytes
        self.x = torch.empty((self.replicas,) + tuple(one.shape), dtype=tdt, device=dev)
        self.x[:] = one
        self.rl = None if row_len is None else torch.from_numpy(row_len).to(dev)
        self.out_idx = torch.empty((c["rows"], c["k"]), dtype=torch.int32, device=dev)
        self.out_val = torch.empty((c["rows"], c["k"]), dtype=tdt, device=dev)
        self.lr0, self.lr1 = local_rows if local_rows is not None else (0, c["rows"])
        self.rows = self.lr1 - self.lr0
        self.read_bytes = workloads.algorithmic_bytes(
            name, row_len=None if row_len is None else row_len[self.lr0:self.lr1], rows=self.rows)
        self.plan = ds.ds_topk_plan(self.x.data_ptr(), self.code, max(self.rows, 1), c["N"],
                                    c["k"], c["B"], c["B2"], 0)
        # one eager call first: attribute set-up and cluster checks happen outside any capture
        self.launch(0, torch.cuda.current_stream(dev).cuda_stream)
        torch.cuda.synchronize(dev)

    def launch(self, i, stream_handle):
        c = self.c
        lib = self.ds.load_library()
        import ctypes
        a, b = self.lr0, self.lr1
        rc = lib.ds_topk(self.x[i % self.replicas, a:b].data_ptr(), self.code, b - a,
                         None if self.rl is None else self.rl[a:b].data_ptr(), c["N"], c["k"],
                         c["B"], c["B2"], ctypes.c_uint64(SEED), self.out_idx[a:b].data_ptr(),
                         self.out_val[a:b].data_ptr(), stream_handle)
        if rc != 0:
            raise self.ds.DSError(rc, "ds_topk", self.ds.ds_last_error_detail())


class LongRowWorkload:
    """One long row (ds_topk_long_row): replicas of the row and the launch
    closure (three kernels per call: pieces, piece results, index gather)."""

    def __init__(self, dev, torch, ds, l2_bytes):
        self.c = c = workloads.LONG_ROW
        self.name = LONG_ROW_NAME
        self.ds = ds
        bits, _ = workloads.generate(1, c["N"], c["dtype"], c["kind"], c["seed"])
        one = torch.from_numpy(bits.reshape(-1).view(np.int32)).to(dev).view(torch.float32)
        del bits
        nbytes = one.numel() * 4
        self.replicas = int(max(2, math.ceil(4 * l2_bytes / nbytes)))
        self.l2_defeated = self.replicas * nbytes >= 4 * l2_bytes
        self.x = torch.empty((self.replicas, c["N"]), dtype=torch.float32, device=dev)
        self.x[:] = one
        del one
        self.rows = 1
        self.esz = 4
        self.read_bytes = workloads.algorithmic_bytes(c)
        self.ws_bytes, self.piece_len, self.pieces = ds.ds_topk_long_row_workspace(
            ds.DS_FP32, c["N"], c["k"], c["B"], c["B2"], plan=True)
        self.plan = {"entry_point": "ds_topk_long_row", "pieces": self.pieces,
                     "piece_len": self.piece_len, "workspace_bytes": self.ws_bytes,
                     "kernels_per_call": 3}
        self.ws = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=dev)
        self.out_idx = torch.empty(c["k"], dtype=torch.int32, device=dev)
        self.out_val = torch.empty(c["k"], dtype=torch.float32, device=dev)
        self.launch(0, torch.cuda.current_stream(dev).cuda_stream)
        torch.cuda.synchronize(dev)
        ref = torch.topk(self.x[0], c["k"], largest=True, sorted=True).values
        self.values_match_torch = bool(torch.equal(ref, self.out_val))

    def launch(self, i, stream_handle):
        import ctypes
        c = self.c
        lib = self.ds.load_library()
        rc = lib.ds_topk_long_row(self.x[i % self.replicas].data_ptr(), self.ds.DS_FP32, c["N"],
                                  c["k"], c["B"], c["B2"], ctypes.c_uint64(SEED),
                                  self.ws.data_ptr(), self.ws_bytes, self.out_idx.data_ptr(),
                                  self.out_val.data_ptr(), stream_handle)
        if rc != 0:
            raise self.ds.DSError(rc, "ds_topk_long_row", self.ds.ds_last_error_detail())


def time_long_row(torch, ds, dev, l2, steps, warmup, peak, burn_seconds):
    """The long-row workload: ds_topk_long_row against torch.topk (context)."""
    wl = LongRowWorkload(dev, torch, ds, l2)
    n = min(steps, 50)
    ms = time_steps(torch, wl, n, warmup, burn_seconds=burn_seconds)
    us = 1e3 * ms / n
    gbs = wl.read_bytes / (us * 1e-6) / 1e9
    x0 = wl.x[0]
    for _ in range(2):
        torch.topk(x0, wl.c["k"], largest=True, sorted=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(5):
        torch.topk(wl.x[i % wl.replicas], wl.c["k"], largest=True, sorted=True)
    e1.record()
    e1.synchronize()
    out = {"workload": wl.c["desc"], "entry_point": "ds_topk_long_row", "us_per_call": us,
           "rows_per_s": 1.0 / (us * 1e-6), "gbs": gbs, "frac_of_measured_hbm": gbs / peak,
           "algorithmic_bytes": wl.read_bytes, "pieces": wl.pieces, "piece_len": wl.piece_len,
           "workspace_bytes": wl.ws_bytes, "kernels_per_call": 3,
           "l2_defeated": wl.l2_defeated, "values_match_torch_topk": wl.values_match_torch,
           "torch_topk": {"us_per_call": e0.elapsed_time(e1) * 1e3 / 5, "timing": "eager"}}
    del wl
    torch.cuda.empty_cache()
    return out


def capture_graph(torch, wl, n, first):
    """A CUDA graph of n launches starting at replica index `first`."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(n):
            wl.launch(first + i, h)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_steps(torch, wl, steps, warmup, dist=None, burn_seconds=0.5):
    """Device time of exactly `steps` launches (graph replays), max over ranks."""
    per_graph = wl.replicas
    full, rest = divmod(steps, per_graph)
    g_full = capture_graph(torch, wl, per_graph, 0) if full else None
    g_rest = capture_graph(torch, wl, rest, 0) if rest else None
    stream = torch.cuda.current_stream()
    # warm-up: W launches, then at least ~0.5 s of back-to-back graphs
    h = stream.cuda_stream
    for i in range(warmup):
        wl.launch(i, h)
    torch.cuda.synchronize()
    t_end = time.perf_counter() + burn_seconds
    g_warm = g_full or g_rest
    while time.perf_counter() < t_end:
        g_warm.replay()
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("deepselect timed steps: %s" % wl.name)
    start.record(stream)
    for _ in range(full):
        g_full.replay()
    if rest:
        g_rest.replay()
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if dist is not None:
        dist.barrier()
    ms = start.elapsed_time(end)
    ms, _ = reduce_over_ranks(ms, 0, dist, device="cuda")
    return ms


def time_e2e(torch, ds, wl, steps):
    """ds_topk_host from pinned host buffers, synchronised every step."""
    c = wl.c
    tdt = wl.x.dtype
    host_dtype = torch.int32 if c["dtype"] == "fp32" else torch.int16
    x_host = torch.from_numpy(wl.bits.view(np.int32 if c["dtype"] == "fp32" else np.int16)).pin_memory()
    rl_host = None if wl.row_len_np is None else torch.from_numpy(wl.row_len_np).pin_memory()
    oi_host = torch.empty((c["rows"], c["k"]), dtype=torch.int32).pin_memory()
    ov_host = torch.empty((c["rows"], c["k"]), dtype=host_dtype).pin_memory()
    x_dev = torch.empty((c["rows"], c["N"]), dtype=tdt, device="cuda")
    rl_dev = None if rl_host is None else torch.empty(c["rows"], dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def one():
        ds.ds_topk_host(x_host.data_ptr(), wl.code, c["rows"],
                        None if rl_host is None else rl_host.data_ptr(), c["N"], c["k"], c["B"],
                        c["B2"], SEED, oi_host.data_ptr(), ov_host.data_ptr(), x_dev.data_ptr(),
                        None if rl_dev is None else rl_dev.data_ptr(), wl.out_idx.data_ptr(),
                        wl.out_val.data_ptr(), stream)

    for _ in range(3):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    dt = time.perf_counter() - t0
    h2d = c["rows"] * c["N"] * wl.esz + (0 if rl_host is None else 4 * c["rows"])
    d2h = c["rows"] * c["k"] * (4 + wl.esz)
    return c["rows"] * steps / dt, h2d, d2h


E2E_DEPTH = 4  # steps in flight in the end-to-end measurement


def time_e2e_pipelined(torch, ds, wl, steps, depth=2):
    """ds_topk_host_async on `depth` streams with as many staging sets: every
    step copies its input from pinned host memory, selects and copies its
    result back; after enqueuing step i the host waits for step i-depth+1 and
    reads its result, so copies and selections of neighbouring steps overlap."""
    c = wl.c
    tdt = wl.x.dtype
    host_dtype = torch.int32 if c["dtype"] == "fp32" else torch.int16
    x_host = torch.from_numpy(wl.bits.view(np.int32 if c["dtype"] == "fp32" else np.int16)).pin_memory()
    rl_host = None if wl.row_len_np is None else torch.from_numpy(wl.row_len_np).pin_memory()
    streams = [torch.cuda.Stream() for _ in range(depth)]
    sets = []
    for _ in range(depth):
        sets.append(dict(
            oi_host=torch.empty((c["rows"], c["k"]), dtype=torch.int32).pin_memory(),
            ov_host=torch.empty((c["rows"], c["k"]), dtype=host_dtype).pin_memory(),
            x_dev=torch.empty((c["rows"], c["N"]), dtype=tdt, device="cuda"),
            rl_dev=None if rl_host is None else torch.empty(c["rows"], dtype=torch.int32, device="cuda"),
            oi_dev=torch.empty((c["rows"], c["k"]), dtype=torch.int32, device="cuda"),
            ov_dev=torch.empty((c["rows"], c["k"]), dtype=tdt, device="cuda")))
    torch.cuda.synchronize()
    checksum = 0

    def issue(i):
        st, b = streams[i % depth], sets[i % depth]
        ds.ds_topk_host_async(x_host.data_ptr(), wl.code, c["rows"],
                              None if rl_host is None else rl_host.data_ptr(), c["N"], c["k"],
                              c["B"], c["B2"], SEED, b["oi_host"].data_ptr(), b["ov_host"].data_ptr(),
                              b["x_dev"].data_ptr(), None if b["rl_dev"] is None else b["rl_dev"].data_ptr(),
                              b["oi_dev"].data_ptr(), b["ov_dev"].data_ptr(), st.cuda_stream)

    def run(n):
        nonlocal checksum
        for i in range(n):
            issue(i)
            j = i - depth + 1
            if j >= 0:
                streams[j % depth].synchronize()
                checksum += int(sets[j % depth]["oi_host"][0, 0])   # the host reads the result
        for j in range(max(0, n - depth + 1), n):
            streams[j % depth].synchronize()
            checksum += int(sets[j % depth]["oi_host"][0, 0])

    run(4)
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    return c["rows"] * steps / dt


def time_torch_topk(torch, wl, steps):
    """torch.topk(sorted=True) on the same replicas (context only)."""
    c = wl.c
    xs = wl.x
    if wl.rl is not None:  # ragged rows: mask the tails first (not timed)
        xs = wl.x.clone()
        cols = torch.arange(c["N"], device=xs.device)[None, :]
        mask = cols >= wl.rl[:, None]
        xs[:, mask] = float("-inf")
    for i in range(3):
        torch.topk(xs[i % wl.replicas], c["k"], dim=-1, largest=True, sorted=True)
    torch.cuda.synchronize()
    n = min(steps, 200)
    mode = "graph"
    try:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            for i in range(min(n, wl.replicas)):
                torch.topk(xs[i % wl.replicas], c["k"], dim=-1, largest=True, sorted=True)
        torch.cuda.current_stream().wait_stream(s)
        reps = max(1, n // min(n, wl.replicas))
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1) / (reps * min(n, wl.replicas))
    except Exception:
        mode = "eager"
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            torch.topk(xs[i % wl.replicas], c["k"], dim=-1, largest=True, sorted=True)
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1) / n
    return {"rows_per_s": c["rows"] / (ms * 1e-3), "us_per_call": ms * 1e3, "timing": mode}


def run_ours(args, rank, world):
    import torch
    import top_selection_deepselect_gb300 as ds

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    ds.load_library()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_kind = measured_peaks()

    long_row = args.workload == LONG_ROW_NAME
    batch_rows = None
    if long_row:
        wl = LongRowWorkload(dev, torch, ds, l2)
    else:
        rows = workloads.CONFIGS[args.workload]["rows"]
        r0, r1, batch_rows = rank_rows(rank, world, rows, args.scaling)
        # weak: this rank's slice of the batch is a full copy of the workload's
        # rows; strong: it is the rows [r0, r1) of the workload itself
        span = (0, rows) if args.scaling == "weak" else (r0, r1)
        wl = Workload(args.workload, dev, torch, ds, l2, local_rows=span)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    ms = time_steps(torch, wl, args.steps, args.warmup, dist=dist, burn_seconds=args.burn_seconds)
    clocks = sampler.stop() if sampler else None

    ms_per_step = ms / args.steps
    _, total_rows = reduce_over_ranks(0.0, wl.rows * args.steps, dist, device="cuda")
    value = total_rows / (ms * 1e-3)
    achieved = wl.read_bytes / (ms_per_step * 1e-3) / 1e9
    c = wl.c
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": args.scaling, "vs_baseline": None, "dtype": c["dtype"],
        "data": data_desc(args.workload),
        "config": dict(cfg_desc(c, args.workload, wl.plan),
                       l2="inputs rotated over %d device replicas (%.0f MB >= 4x L2 %.0f MB)"
                          % (wl.replicas, wl.replicas * c["rows"] * c["N"] * wl.esz / 1e6,
                             l2 / 1e6),
                       parallelism=("contiguous row ranges of a %d-row batch, one per rank, no "
                                    "exchange" % batch_rows) if world > 1 else "1 GPU"),
        "gpu_launches": args.steps * (3 if long_row else 1),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": None if long_row else profile_traffic(args.workload, kernel_name(wl.plan)),
                     "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": wl.read_bytes,
                     "kernel": None if long_row else kernel_name(wl.plan)},
        "clocks": clocks,
    }
    if long_row:
        line["roofline"]["kernel"] = "ds_topk_long_row call (pieces, piece results, gather)"
        line["e2e"] = None
        line["note"] = ("long-row workload: achieved = the row's bytes / the whole call; no "
                        "end-to-end number or extras")
    if rank == 0 and not long_row:
        e2e_steps = args.e2e_steps or args.steps
        e2e_sync, h2d, d2h = time_e2e(torch, ds, wl, e2e_steps)
        e2e_pipe = time_e2e_pipelined(torch, ds, wl, e2e_steps, depth=E2E_DEPTH)
        line["e2e"] = {"value": e2e_pipe * world, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                       "path": "ds_topk_host_async, %d steps in flight on %d streams (pinned host "
                               "buffers; each step copies its input, selects, copies its result "
                               "back; the host reads every step's result); kernels of different "
                               "steps may run concurrently" % (E2E_DEPTH, E2E_DEPTH),
                       "sync_per_step_value": e2e_sync * world,
                       "sync_per_step_path": "ds_topk_host, synchronised every step"}
    if rank == 0 and world == 1 and not args.no_extras and not long_row:
        line["torch_topk"] = time_torch_topk(torch, wl, args.steps)
        per = {}
        for name in workloads.CONFIG_ORDER:
            w2 = wl if name == args.workload else Workload(name, dev, torch, ds, l2)
            ms2 = time_steps(torch, w2, args.steps, args.warmup, burn_seconds=args.burn_seconds)
            us = 1e3 * ms2 / args.steps
            gbs = w2.read_bytes / (us * 1e-6) / 1e9
            per[name] = {"us_per_call": us, "rows_per_s": w2.rows / (us * 1e-6), "gbs": gbs,
                         "frac_of_measured_hbm": gbs / peak, "frac_of_spec_hbm": gbs / SPEC_HBM_GBS,
                         "l2_defeated": w2.l2_defeated,
                         "algorithmic_bytes": w2.read_bytes, "plan": w2.plan,
                         "torch_topk": time_torch_topk(torch, w2, args.steps)}
            if name != args.workload:
                rate, dt, done, step_rows = oracle_rows_per_s(
                    name, seconds=args.cpu_seconds_per_config, rows_per_step=1)
                per[name]["cpu_baseline"] = {
                    "value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                    "sample": "%d rows of %s in %.1f s (rows cycled), single thread"
                              % (done * step_rows, name, dt)}
            if w2 is not wl:
                del w2
                torch.cuda.empty_cache()
        line["per_config"] = per
        line["long_row"] = time_long_row(torch, ds, dev, l2, args.steps, args.warmup, peak,
                                         args.burn_seconds)
        rate, dt, done, step_rows = oracle_rows_per_s(args.workload, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": "%d rows of %s in %.1f s (rows cycled), single thread"
                                          % (done * step_rows, args.workload, dt),
                                "host": host_cpu()}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, _ = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world)


if __name__ == "__main__":
    main()

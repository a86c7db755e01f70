#!/usr/bin/env python3
"""Benchmark of the QSA indexer step (score + exact top-k) on GB300.

One step = one qsa_select_paged_tokens call over one batch, inputs resident
in HBM.  Default workload: the last 1,616-row prefill chunk of a
184,320-token context (46,080 compressed positions, 4 heads x 128, top-2,048,
64-token pages).  Prints one JSON line (rank 0).

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

--impl reference times the CPU oracle (the only reference implementation of
this step) on the host cores, on a bounded sample of rows per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_attention_select_gb300 import workloads as W  # noqa: E402

METRIC = "indexer rows/s (score + exact top-k) and % of roofline on 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[key] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                out["source"] = "measured"
                return out
        except Exception:
            pass
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def algorithmic(wl):
    """Scoring FLOPs and compulsory bytes of one step (per the step's definition)."""
    pairs = wl.visible_pairs
    H, D = wl.heads, 128
    flops = 2.0 * H * D * pairs
    P = wl.k_cache.shape[1]
    pages = int(np.sum((wl.req_positions.astype(np.int64) + P - 1) // P))
    key_bytes = pages * P * D * 2
    q_bytes = wl.q.nbytes + wl.w.nbytes + wl.row_req.nbytes + wl.row_visible.nbytes
    logit_bytes = 4 * pairs
    idx_bytes = wl.rows * wl.k * 4
    return dict(flops=flops, key_bytes=key_bytes, q_bytes=q_bytes, logit_bytes=logit_bytes,
                idx_bytes=idx_bytes, bytes=key_bytes + q_bytes + logit_bytes + idx_bytes,
                pairs=pairs)


class ClockSampler:
    """SM clock and throttle-reason samples taken while the timed region runs.

    Reads NVML through ctypes every ~0.5 ms from a background thread (the
    timed region of a short run lasts a few milliseconds); falls back to
    nvidia-smi at 200 ms where libnvidia-ml cannot be loaded.  Read-only:
    no clock or other GPU setting is changed."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clocks-event-reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.nvml = None
        self.samples = []
        self.stop_flag = threading.Event()

    def _nvml_open(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return None
        return lib, h

    def _poll(self):
        import ctypes
        lib, h = self.nvml
        mhz, mx, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0            # NVML_CLOCK_SM
            ok = ok and lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
            ok = ok and get_reasons(h, ctypes.byref(reasons)) == 0
            if ok:
                self.samples.append((mhz.value, mx.value, reasons.value))
            time.sleep(0.0005)

    def start(self):
        try:
            self.nvml = self._nvml_open()
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.nvml is not None:
            self.stop_flag.set()
            self.t.join(timeout=2)
            if not self.samples:
                return None
            reasons = set()
            for _, _, bits in self.samples:
                for bit, name in self.REASONS.items():
                    if bits & bit:
                        reasons.add(name)
            return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                    "sm_max_mhz": max(s[1] for s in self.samples), "reasons": sorted(reasons),
                    "samples": len(self.samples), "source": "nvml, every ~0.5 ms"}
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, every 200 ms"}


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_rows_per_s(wl, nrows: int, threads: int = 0):
    """Time the oracle (as it stands) on the first nrows rows of the workload."""
    import oracle
    rows = np.linspace(0, wl.rows - 1, num=min(nrows, wl.rows)).astype(np.int64)
    t0 = time.perf_counter()
    oracle.select_paged_tokens(wl.q[rows], wl.w[rows], wl.k_cache, wl.block_table,
                               wl.row_req[rows], wl.row_visible[rows], wl.k, ld=wl.ld,
                               nthreads=threads)
    dt = time.perf_counter() - t0
    return len(rows) / dt, len(rows), dt


def cpu_baseline(wl, budget_s: float = 12.0):
    import oracle
    cores = oracle.max_threads()
    # calibrate on a handful of rows, then size the sample to the budget
    rps, n, dt = oracle_rows_per_s(wl, max(cores, 4))
    n2 = int(min(wl.rows, max(n, rps * budget_s * 0.8)))
    if n2 > n:
        rps, n, dt = oracle_rows_per_s(wl, n2)
    return {"value": rps, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {wl.rows} rows of {wl.name} (evenly spaced), all visible "
                      f"positions each, {dt:.1f} s on {cores} threads"}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    wl = W.CONFIGS[args.workload]()
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    per_step = max(4, 2 * cores)
    rps0, _, dt0 = oracle_rows_per_s(wl, per_step)
    # keep the whole --steps/--warmup run within a few minutes
    budget = 150.0 / max(1, args.steps + args.warmup)
    if dt0 > budget:
        per_step = max(1, int(per_step * budget / dt0))
    for _ in range(args.warmup):
        oracle_rows_per_s(wl, per_step)
    times, rows = [], 0
    t_all = time.perf_counter()
    for _ in range(args.steps):
        _, n, dt = oracle_rows_per_s(wl, per_step)
        times.append(dt)
        rows += n
    total = time.perf_counter() - t_all
    value = rows / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "rows": wl.rows, "k": wl.k, "heads": wl.heads,
                   "sample_rows_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} evenly spaced rows of {wl.rows} per step"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def capture_step(args, qsa, step, outputs):
    """The timed loop replays one call captured as a CUDA graph: the same
    launches on the same resident inputs, one graph launch of host work per
    step, so the host never leaves the GPU idle inside a timed step.  A capture
    that fails, or a replay whose outputs differ from an eager call's, falls
    back to eager calls.  Returns (launch mode, step function)."""
    import torch

    if args.eager:
        return "eager", step
    ref = [t.clone() for t in outputs]                    # the last eager call's results
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for t in outputs:
            t.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        ok = qsa.get_device_status() == qsa.QSA_OK and all(torch.equal(a, b) for a, b in zip(outputs, ref))
    except Exception as e:                                # noqa: BLE001 (any capture failure: eager)
        torch.cuda.synchronize()
        qsa.get_device_status()
        return f"eager (graph capture failed: {type(e).__name__})", step
    if not ok:
        return "eager (graph replay differed)", step
    return "cuda_graph", graph.replay


def run_ours(args, ws, rank, local):
    import torch

    from block_sparse_attention_select_gb300 import qsa

    qsa.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = W.CONFIGS[args.workload]()
    alg = algorithmic(wl)
    peaks = load_peaks()

    q = torch.from_numpy(wl.q).to(dev)
    w = torch.from_numpy(wl.w).to(dev)
    rr = torch.from_numpy(wl.row_req).to(dev)
    rv = torch.from_numpy(wl.row_visible).to(dev)
    keys = qsa.PagedKeys(torch.from_numpy(wl.k_cache).to(dev), torch.from_numpy(wl.block_table).to(dev))
    out_idx = torch.empty((wl.rows, wl.k), dtype=torch.int32, device=dev)
    out_val = torch.empty((wl.rows, wl.k), dtype=torch.float32, device=dev)
    wsb = qsa.alloc_workspace(wl.rows, keys.max_len, wl.k, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    qsa.set_config(qsa.QSA_CFG_PATH, {"auto": 0, "dense": 1, "filter": 2}[args.path])
    stream = torch.cuda.current_stream()

    def step():
        # the stream current at the call: the capture stream while a graph is captured
        qsa.select_paged_tokens(q, w, keys, rr, rv, wl.k, out_idx, out_val, wsb, torch.cuda.current_stream())

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert qsa.get_device_status() == qsa.QSA_OK
    launches_per_step = qsa.last_launch_count()
    launch, timed_step = capture_step(args, qsa, step, (out_idx, out_val))

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for a, b in ev:
        flush.zero_()                                     # L2 flushed between steps
        a.record(stream)
        timed_step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)

    # per-kernel breakdown: a separate, shorter pass in which the library
    # brackets every launch with CUDA events on its stream (kept out of the
    # timed region above, whose events bracket whole steps only)
    qsa.set_config(qsa.QSA_CFG_KERNEL_TIMING, 1)
    qsa.kernel_times()                                   # drop anything pending
    n_kt = max(1, min(args.steps, 200))
    for _ in range(n_kt):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    kt = qsa.kernel_times()
    qsa.set_config(qsa.QSA_CFG_KERNEL_TIMING, 0)
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)

    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms_local, ws)
    value = wl.rows * ws / (ms / 1e3)

    # dominant kernel: the scorer launch with the largest total time
    dom = max(kt.items(), key=lambda kv: kv[1][0])
    dom_name, (dom_ms_total, dom_n) = dom
    dom_ms = dom_ms_total / max(1, dom_n)
    if dom_name.startswith("score"):
        # the scorer is bound by its FLOPs at the tensor peak or by its key and
        # query reads at the HBM peak, whichever takes longer (decode batches
        # read ~285 MB of keys for ~1 GFLOP)
        frac_work = 1.0 / 16 if dom_name == "score_sample" else 1.0
        kbytes = (alg["key_bytes"] + alg["q_bytes"]) * frac_work
        if alg["flops"] * frac_work / (peaks["bf16_tflops"] * 1e12) >= kbytes / (peaks["hbm_gbs"] * 1e9):
            bound, unit = "tensor", "TFLOP/s"
            work = alg["flops"] * frac_work
            achieved = work / (dom_ms / 1e3) / 1e12
            peak = peaks["bf16_tflops"]      # burst figure: the kernel runs for microseconds
        else:
            bound, unit = "hbm", "GB/s"
            work = kbytes
            achieved = work / (dom_ms / 1e3) / 1e9
            peak = peaks["hbm_gbs"]
    else:
        bound, unit = "hbm", "GB/s"
        work = alg["logit_bytes"] + alg["idx_bytes"]
        achieved = work / (dom_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
    t_flop = alg["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_mem = alg["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_roof = max(t_flop, t_mem)
    roof_traffic = recorded_traffic(wl.name, dom_name)

    # end to end through the public API: host inputs in, host result out
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, wl, qsa, keys, stream, dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl)

    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": wl.name, "rows": wl.rows, "positions_max": int(wl.row_visible.max()),
                   "visible_pairs": alg["pairs"], "k": wl.k, "heads": wl.heads, "head_dim": 128,
                   "page_positions": int(wl.k_cache.shape[1]), "path": args.path,
                   "l2": "flushed between steps (512 MiB write)", "launch": launch,
                   "accumulate": "f32", "median_ms": statistics.median(step_ms)},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": roof_traffic, "kernel": dom_name,
                     "kernel_ms": dom_ms, "peak_source": peaks["source"]},
        "step_roofline": {"t_roof_us": t_roof * 1e6, "t_flop_us": t_flop * 1e6,
                          "t_mem_us": t_mem * 1e6, "frac": t_roof / (ms / 1e3),
                          "gflop": alg["flops"] / 1e9, "mbytes": alg["bytes"] / 1e6,
                          "peak_source": peaks["source"]},
        "kernels_ms_per_step": {k: v[0] / n_kt for k, v in kt.items()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# the sources each measured kernel is compiled from: its own file and the
# shared headers (a change anywhere else leaves its recorded traffic valid)
KERNEL_SOURCES = {
    "score": ("qsa_score.cu", "qsa_device.cuh", "qsa_internal.h"),
    "select": ("qsa_select.cu", "qsa_device.cuh", "qsa_internal.h"),
    "produce": ("qsa_produce.cu", "qsa_device.cuh", "qsa_internal.h"),
    "attend": ("qsa_attend.cu", "qsa_device.cuh", "qsa_internal.h"),
}


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` on `workload` from the ncu record in
    profiles/traffic.json, or None when there is none or the kernel's sources
    have changed since it was taken."""
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tr_path):
        return None
    try:
        ent = json.load(open(tr_path)).get(workload, {}).get(kernel)
    except Exception:
        return None
    if ent and ent.get("kernel_rev") == kernel_revision(kernel):
        return ent["bytes_per_launch"]
    return None


def kernel_revision(kernel: str) -> str:
    """Hash of the sources of `kernel` (a kernel-times name such as
    score_filter or select_cand, or produce)."""
    import hashlib
    files = KERNEL_SOURCES.get(kernel.split("_")[0])
    if files is None:
        return ""                                         # no recorded traffic for this kernel
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "block_sparse_attention_select_gb300", "csrc")
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:12]


def measure_e2e(args, wl, qsa, keys_dev, stream, dev):
    """End to end through the public call: every step copies its inputs from
    pinned host memory, runs qsa_select_paged_tokens and copies its indices
    back to pinned host memory.  Steps are pipelined the way a serving loop
    would run them: the copies ride their own streams and overlap the previous
    step's compute (two device input and output sets); every copy still
    happens inside the timed region."""
    import torch
    names = ("q", "w", "row_req", "row_visible", "k_cache", "block_table")
    host = {n: torch.from_numpy(getattr(wl, n)).pin_memory() for n in names}
    dbuf = [{n: torch.empty_like(t, device=dev) for n, t in host.items()} for _ in range(2)]
    keys = [qsa.PagedKeys(b["k_cache"], b["block_table"]) for b in dbuf]
    out = [torch.empty((wl.rows, wl.k), dtype=torch.int32, device=dev) for _ in range(2)]
    out_host = [torch.empty((wl.rows, wl.k), dtype=torch.int32).pin_memory() for _ in range(2)]
    wsb = qsa.alloc_workspace(wl.rows, keys_dev.max_len, wl.k, dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host[0].numel() * out_host[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def one(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(comp_done[b])          # the step that last used these inputs has run
            for n in names:
                dbuf[b][n].copy_(host[n], non_blocking=True)
            in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if started[b]:
            stream.wait_event(out_done[b])             # its indices have left the device
        qsa.select_paged_tokens(dbuf[b]["q"], dbuf[b]["w"], keys[b], dbuf[b]["row_req"], dbuf[b]["row_visible"],
                                wl.k, out[b], None, wsb, stream, with_values=False)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            out_host[b].copy_(out[b], non_blocking=True)
            out_done[b].record(s_out)
        started[b] = True

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    n = max(6, min(args.steps, 500))
    t0 = time.perf_counter()
    for i in range(n):
        one(i)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / n
    return {"value": wl.rows / dt, "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3,
            "pipelined": "copies on their own streams, overlapping the previous step's compute"}


PRODUCE_METRIC = "index-key producer keys/s (pool + RMSNorm + RoPE + paged store) on 1 GB300"


def keys_written(pos_start: int, n_tokens: int, window: int) -> int:
    """Index keys one request's call stores: the blocks of four tokens that end
    among the new tokens [pos_start, pos_start + n_tokens) and whose pooling
    window, clipped at position 0, starts at or after pos_start."""
    first = (pos_start + 3) // 4                  # first block ending at or after pos_start
    last = (pos_start + n_tokens) // 4 - 1        # last block ending before the end
    n = 0
    for i in range(first, last + 1):
        if max(0, 4 * i + 4 - window) >= pos_start:
            n += 1
    return n


def produce_bytes(inp):
    """Algorithmic bytes of one producer call: every token key (and pooling
    logit) read once, per stored key its RoPE table row, its block-table entry
    and the 256-byte FP16 key written."""
    nkeys = sum(keys_written(int(inp.pos_start[b]), int(inp.seq_start[b + 1] - inp.seq_start[b]), inp.window)
                for b in range(len(inp.pos_start)))
    read = inp.tokens * 256 + (inp.tokens * 4 if inp.pool_logit is not None else 0)
    per_key = inp.rope_dim * 4 + 4 + 256
    return nkeys, read + nkeys * per_key


def run_produce(args, ws, rank, local):
    import torch

    from block_sparse_attention_select_gb300 import qsa

    qsa.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.PRODUCER_CONFIGS[args.producer_workload](window=args.window, logits=args.window == 8)
    nkeys, alg_bytes = produce_bytes(inp)
    peaks = load_peaks()
    x = torch.from_numpy(inp.x).to(dev)
    pl = torch.from_numpy(inp.pool_logit).to(dev) if inp.pool_logit is not None else None
    ss = torch.from_numpy(inp.seq_start).to(dev)
    ps = torch.from_numpy(inp.pos_start).to(dev)
    g = torch.from_numpy(inp.norm_weight).to(dev)
    kc = torch.from_numpy(inp.k_cache).to(dev)
    keys = qsa.PagedKeys(kc, torch.from_numpy(inp.block_table).to(dev))
    nb = int(((inp.pos_start.astype(np.int64) + np.diff(inp.seq_start)) // 4).max()) + 1
    tab = qsa.rope_table(nb, inp.rope_dim, inp.theta)       # built once per model, not per step
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        qsa.index_key_produce(x, ss, ps, inp.max_tokens, g, tab, keys, pool_logit=pl, eps=inp.eps,
                              rope_dim=inp.rope_dim, window=inp.window, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for a, b in ev:
        flush.zero_()                                     # inputs fit in L2: flush between steps
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), ws)
    achieved = alg_bytes / (ms / 1e3) / 1e9              # one launch per step
    e2e = None
    if not args.no_e2e:
        hx = torch.from_numpy(inp.x).pin_memory()
        hl = torch.from_numpy(inp.pool_logit).pin_memory() if inp.pool_logit is not None else None
        hout = torch.empty(kc.shape, dtype=kc.dtype).pin_memory()
        n_e = max(3, min(args.steps, 50))
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(n_e):
            x.copy_(hx, non_blocking=True)
            if hl is not None:
                pl.copy_(hl, non_blocking=True)
            step()
            hout.copy_(kc, non_blocking=True)
            torch.cuda.synchronize()
        el = (time.perf_counter() - t) / n_e
        h2d = hx.numel() * 2 + (hl.numel() * 4 if hl is not None else 0)
        e2e = {"value": nkeys / el, "unit": "keys/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hout.numel() * 2, "ms_per_step": el * 1e3}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        from oracle import producer as P
        t = time.perf_counter()
        _, done = P.produce(inp.x, inp.pool_logit, inp.seq_start, inp.pos_start, inp.norm_weight, inp.eps,
                            inp.rope_dim, inp.theta, inp.window, inp.k_cache, inp.block_table)
        el = time.perf_counter() - t
        cpu = {"value": len(done) / el, "unit": "keys/s", "cores": 1, "kind": "oracle",
               "sample": f"all {len(done)} keys of {inp.name} (numpy float64, one thread), {el:.1f} s"}
    traffic = recorded_traffic(f"{inp.name}_w{inp.window}", "produce")
    line = {
        "metric": PRODUCE_METRIC, "value": nkeys * ws / (ms / 1e3), "unit": "keys/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 in / f32 math / f16 out", "data": "synthetic",
        "config": {"workload": f"{inp.name}_w{inp.window}", "tokens": inp.tokens, "keys": nkeys,
                   "window": inp.window, "pool_logits": inp.pool_logit is not None, "rope_dim": inp.rope_dim,
                   "page_positions": int(inp.k_cache.shape[1]), "l2": "flushed between steps (512 MiB write)",
                   "median_ms": statistics.median(step_ms)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": "produce",
                     "kernel_ms": ms, "algorithmic_bytes": alg_bytes, "peak_source": peaks["source"]},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


ATTEND_METRIC = "sparse-attention consumer rows/s (raw tokens of the selected positions, GQA 24/2 x 256) on 1 GB300"


def run_attend(args, ws, rank, local):
    import torch

    from block_sparse_attention_select_gb300 import qsa

    qsa.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    # the prefill chunk of the indexer bench: 1,616 query rows at the end of a
    # 184,320-token context, each attending its top-2,048 positions' raw tokens
    inp = W.make_consumer_inputs("consumer_1616rows_ctx184320_k2048", seed=31, ctx_tokens=[184_320],
                                 rows_per_req=[1616], k=2048)
    R, hq, D = inp.q.shape
    hkv = inp.k_cache.shape[2]
    toks = sum(4 * int((row >= 0).sum()) + (int(t) + 1 - 4 * ((int(t) + 1) // 4))
               for row, t in zip(inp.sel, inp.row_token))
    flops = 4.0 * hq * D * toks                          # QK and PV, 2 FLOP per multiply-add
    gathered = 2.0 * toks * hkv * D * 2                  # K and V lines read through the block table
    peaks = load_peaks()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q, kc, vc, bt = t(inp.q), t(inp.k_cache), t(inp.v_cache), t(inp.block_table)
    rr, rt, sel = t(inp.row_req), t(inp.row_token), t(inp.sel)
    out = torch.empty((R, hq, D), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        qsa.sparse_attention(q, kc, vc, bt, rr, rt, sel, out=out, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), ws)
    achieved = flops / (ms / 1e3) / 1e12
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        from oracle import consumer as C
        n_s = 4
        t0 = time.perf_counter()
        C.sparse_attention(inp.q[:n_s], inp.k_cache, inp.v_cache, inp.block_table, inp.row_req[:n_s],
                           inp.row_token[:n_s], inp.sel[:n_s])
        el = time.perf_counter() - t0
        cpu = {"value": n_s / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
               "sample": f"the first {n_s} rows of {R} (numpy float64, one thread), {el:.1f} s"}
    line = {
        "metric": ATTEND_METRIC, "value": R * ws / (ms / 1e3), "unit": "rows/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 in / f32 math / f32 out", "data": "synthetic",
        "config": {"workload": inp.name, "rows": R, "q_heads": hq, "kv_heads": hkv, "head_dim": D, "k": 2048,
                   "tokens_attended": toks, "gathered_gb": gathered / 1e9,
                   "l2": "flushed between steps (512 MiB write)", "median_ms": statistics.median(step_ms)},
        # QK and PV are contractions: measured against the dense FP16 tensor peak;
        # the gathered K / V lines (~12 FLOP per byte, each row reading its own
        # tokens from a cache larger than L2) give the memory-side bound beside it
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": recorded_traffic(inp.name, "attend"), "kernel": "attend", "kernel_ms": ms,
                     "gathered_gb_per_s": gathered / (ms / 1e3) / 1e9, "peak_source": peaks["source"]},
        "gather_bound": {"bytes": gathered, "t_hbm_ms": gathered / (peaks["hbm_gbs"] * 1e9) * 1e3,
                         "t_tensor_ms": flops / (peaks["bf16_tflops"] * 1e12) * 1e3,
                         "frac_of_hbm": gathered / (ms / 1e3) / (peaks["hbm_gbs"] * 1e9)},
        "cpu_baseline": cpu,
        "e2e": None,
        "gpu_launches": args.steps,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


BLOCKS_METRIC = "block-scorer rows/s (per-head 128-token block max + exact top-k) on 1 GB300"


def run_blocks(args, ws, rank, local):
    import torch

    from block_sparse_attention_select_gb300 import qsa

    qsa.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.block_scorer_bench()
    R, H, D = inp.q.shape
    tokens = int(np.sum(inp.row_token.astype(np.int64) + 1))
    flops = 2.0 * D * H * tokens                       # every visible token's dot product per head
    peaks = load_peaks()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q, kc, bt, rr, rt = t(inp.q), t(inp.k_cache), t(inp.block_table), t(inp.row_req), t(inp.row_token)
    oi = torch.empty((R, H, inp.k), dtype=torch.int32, device=dev)
    ov = torch.empty((R, H, inp.k), dtype=torch.float32, device=dev)
    wsb = torch.empty(int(qsa.load().qsa_block_select_workspace_bytes(R, H, int(bt.shape[1]), inp.k)),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        qsa.block_select(q, kc, bt, rr, rt, inp.k, oi, ov, wsb, stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    launches = qsa.last_launch_count()
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), ws)
    # per-kernel times (a separate pass with events around every launch)
    qsa.set_config(qsa.QSA_CFG_KERNEL_TIMING, 1)
    qsa.kernel_times()
    n_kt = max(1, min(args.steps, 100))
    for _ in range(n_kt):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    kt = qsa.kernel_times()
    qsa.set_config(qsa.QSA_CFG_KERNEL_TIMING, 0)
    score_ms = kt.get("score_blocks", (ms * n_kt, n_kt))[0] / n_kt
    achieved = flops / (score_ms / 1e3) / 1e12
    e2e = None
    if not args.no_e2e:
        hq, hk = torch.from_numpy(inp.q).pin_memory(), torch.from_numpy(inp.k_cache).pin_memory()
        hout = torch.empty((R, H, inp.k), dtype=torch.int32).pin_memory()
        n_e = max(3, min(args.steps, 50))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e):
            q.copy_(hq, non_blocking=True)
            kc.copy_(hk, non_blocking=True)
            qsa.block_select(q, kc, bt, rr, rt, inp.k, oi, None, wsb, stream, with_values=False)
            hout.copy_(oi, non_blocking=True)
            torch.cuda.synchronize()
        el = (time.perf_counter() - t0) / n_e
        e2e = {"value": R * ws / el, "unit": "rows/s", "h2d_bytes_per_step": hq.numel() * 2 + hk.numel() * 2,
               "d2h_bytes_per_step": hout.numel() * 4, "ms_per_step": el * 1e3}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        from oracle import block_scorer as BS
        n_s = 4
        rows = np.linspace(0, R - 1, n_s).astype(np.int64)
        t0 = time.perf_counter()
        BS.select_blocks(inp.q[rows], inp.k_cache, inp.block_table, inp.row_req[rows], inp.row_token[rows], inp.k)
        el = time.perf_counter() - t0
        cpu = {"value": n_s / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
               "sample": f"{n_s} evenly spaced rows of {R} (numpy float64, one thread), {el:.1f} s"}
    line = {
        "metric": BLOCKS_METRIC, "value": R * ws / (ms / 1e3), "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": inp.name, "rows": R, "kv_heads": H, "head_dim": D, "k_blocks": inp.k,
                   "block_tokens": 128, "visible_tokens": tokens, "l2": "flushed between steps (512 MiB write)",
                   "accumulate": "f32", "median_ms": statistics.median(step_ms)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": recorded_traffic(inp.name, "score_blocks"), "kernel": "score_blockrows",
                     "kernel_ms": score_ms, "gflop": flops / 1e9, "peak_source": peaks["source"]},
        "kernels_ms_per_step": {k: v[0] / n_kt for k, v in kt.items()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.CONFIGS), default="bench")
    ap.add_argument("--path", choices=["auto", "dense", "filter"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager calls instead of a captured graph of one call")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--op", choices=["select", "produce", "attend", "blocks"], default="select",
                    help="select: the indexer step (default); produce: the index-key producer; "
                         "attend: the sparse-attention consumer; blocks: the M3-style block scorer")
    ap.add_argument("--producer-workload", choices=sorted(W.PRODUCER_CONFIGS), default="context")
    ap.add_argument("--window", type=int, choices=[4, 8], default=4)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    ws, rank, local = dist_setup()
    if args.op == "blocks":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the block scorer's reference arm is the "
                                  "oracle, reported as cpu_baseline in the blocks line"}), flush=True)
        else:
            run_blocks(args, ws, rank, local)
    elif args.op == "attend":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the consumer's reference arm is the "
                                  "oracle, reported as cpu_baseline in the attend line"}), flush=True)
        else:
            run_attend(args, ws, rank, local)
    elif args.op == "produce":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the producer's reference arm is the "
                                  "oracle, reported as cpu_baseline in the produce line"}), flush=True)
        else:
            run_produce(args, ws, rank, local)
    elif args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

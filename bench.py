"""Benchmark: RNN-T joint + output layer + transducer loss, forward + backward.

One step = one training step over one batch of the synthetic workload (every
row of the hot path: validation, projections, the tiled joint/output/LSE
forward, alpha/beta, the tiled recompute backward, the encoder gradients),
through rnnt_fwd_bwd (`--api separate`: rnnt_fwd then rnnt_bwd).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload audio40] [--impl reference]

The default workload is the 40 s, batch-1024 configuration (B=1024, T=1000,
U=100, H=512, V=4096, bf16, tiled); the other workloads of
asr_tiled_tanh_gb300/synthetic.py are parity-test cases that can be timed the
same way with --workload.

Prints one JSON line (rank 0).  `value` is lattice cells B*T*(U+1) per second
over all ranks with inputs already in HBM; `e2e` is the same metric through
the C ABI with host buffers: every timed step copies its batch (hA, hL,
labels, lengths) from pinned host memory to the device and reads its losses
back; the parameters and their gradients stay on the device, where a training
step keeps them.  Each rank runs its own batch (weak
scaling, data-parallel): with N ranks every step ends with one all-reduce
(sum) of the parameter gradients, the only exchange the path has.  `--gpus N`
starts N processes itself when no launcher did.  L2 is flushed (256 MiB write)
before every timed step, outside the step's events.

When the library reports the plan capturable (rnnt_graph_capturable: the
whole lattice fits one chunk, so the calls make no host synchronization), the
timed steps replay a CUDA graph of the step (`config.execution`); `--eager`
launches them one by one instead.  A second, eager run of the same number of
steps with every kernel bracketed by CUDA events on its own stream gives the
per-kernel times (`kernel_shares`, `roofline`) and `gpu_launches`.  A third
eager run times rnnt_fwd and rnnt_bwd apart (`ms_by_phase`: medians of the
forward, the backward and their sum, and the median of the timed steps).  A bf16
workload is then timed once more with the score products on e4m3 tensor cores
(`e4m3_scores`, a secondary line on its own plan; `--no-e4m3-leg` skips it).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RNN-T fwd+bwd lattice cells/s (B*T*(U+1)); peak HBM GB; % bf16 tensor peak"
UNIT = "cells/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _smi_index(cuda_index: int) -> int:
    """nvidia-smi / NVML index of a CUDA device (CUDA_VISIBLE_DEVICES, when it
    lists plain indices, renumbers the devices a process sees)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    if ids and all(x.isdigit() for x in ids) and cuda_index < len(ids):
        return int(ids[cuda_index])
    return cuda_index


class _Nvml:
    """SM clock and clock-event reasons read in-process through the NVIDIA
    management library (the library nvidia-smi itself reads). Read-only."""

    CLOCK_SM = 1
    IDLE = 0x1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) != 0:
            lib.nvmlShutdown()
            raise OSError("no NVML device %d" % index)
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.dev, self.CLOCK_SM, ctypes.byref(mx))
        self.max_mhz = float(mx.value)

    def read(self):
        """(sm MHz, reason bits) or None."""
        ct = self.ct
        mhz, bits = ct.c_uint(0), ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.dev, self.CLOCK_SM, ct.byref(mhz)) != 0:
            return None
        if self.reasons_fn is not None:
            self.reasons_fn(self.dev, ct.byref(bits))
        return float(mhz.value), int(bits.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clocks and throttle reasons during a timed region: an in-process
    NVML poll every 2 ms on a background thread (so that even a region of a
    few milliseconds is covered; `sample_now()` adds one from the caller
    while its queued work runs), plus nvidia-smi every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, poll_s: float = 0.002):
        self.gpu = _smi_index(gpu_index)
        self.poll_s = poll_s
        self.proc = None
        self.nvml = None
        self.nvml_samples = []
        self.lines = []

    def sample_now(self):
        if self.nvml is not None:
            r = self.nvml.read()
            if r is not None:
                self.nvml_samples.append(r)

    def _poll(self):
        while not self._stop.is_set():
            self.sample_now()
            self._stop.wait(self.poll_s)

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        try:
            self.nvml = _Nvml(self.gpu)
        except Exception:
            self.nvml = None
        self._stop = threading.Event()
        self._thread = None
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self.nvml is not None:
            self.nvml.close()
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        """Median SM clock over the samples taken under load (NVML samples
        flagged GPU-idle are left out when others exist), the maximum clock
        and every throttle reason seen active."""
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        n_smi = 0
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            n_smi += 1
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        busy = [s for s in self.nvml_samples if not s[1] & _Nvml.IDLE] or self.nvml_samples
        for mhz, bits in busy:
            sm.append(mhz)
            for bit, n in _Nvml.REASONS.items():
                if bits & bit:
                    reasons.add(n)
        if busy and self.nvml is not None:
            mx.append(self.nvml.max_mhz)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "sources": {"nvml_2ms": len(busy), "nvidia_smi_200ms": n_smi}}


# Algorithmic DRAM bytes per valid lattice position of the memory-bound
# kernels that can dominate a step: the untiled dh pass reads the kept bf16
# scores and the 16-byte posterior record and writes dh over the scores.
KERNEL_BYTES_PER_CELL = {"tc_dh_kept": lambda V: 4 * V + 16}


# Algorithmic tensor work of each tensor-core kernel, per valid lattice
# position, in units of H*V flops (the projections and encoder GEMMs are
# accounted per encoder row instead).
KERNEL_FLOPS_PER_CELL_HV = {"tc_fwd_tiles": 2.0, "tc_bwd_dh": 2.0, "tc_bwd_dz": 2.0,
                            "tc_bwd_dwo": 2.0}
# The kernels whose products run on e4m3 operands with --scores e4m3.
E4M3_KERNELS = ("tc_fwd_tiles", "tc_bwd_dh")


def kernel_source_hash(root: str | None = None) -> str:
    """sha1 of the sources that decide the lattice GEMMs' DRAM traffic, with
    comments and whitespace removed: k_tc.cu (the tensor-core kernels and their
    launches), every header it includes, transitively (tile geometry, the
    workspace layout, the PTX wrappers), and api.cu (the plan: chunk sizes and
    buffer placement).  The ncu traffic figures are only valid for the code
    they were captured from; the other translation units (the alpha/beta
    recursion, the fp32 path, the no-allocation entry point) do not touch the
    GEMMs."""
    import hashlib
    import re
    csrc = os.path.join(root or ROOT, "asr_tiled_tanh_gb300", "csrc")
    todo = [os.path.join(csrc, "k_tc.cu"), os.path.join(csrc, "api.cu")]
    seen = []
    while todo:
        path = os.path.normpath(todo.pop(0))
        if path in seen or not os.path.exists(path):
            continue
        seen.append(path)
        with open(path) as fh:
            for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', fh.read(), flags=re.M):
                todo.append(os.path.join(os.path.dirname(path), inc))
    h = hashlib.sha1()
    for path in sorted(seen, key=os.path.basename):
        h.update(os.path.basename(path).encode())
        with open(path) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:12]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summaries in profiles/ (a line `traffic <kernel> <workload> <bytes> src=<sha>`),
    or None when absent or taken from different kernel source."""
    import glob
    import re
    want = kernel_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(path):
            m = re.match(r"\s*traffic\s+(\S+)\s+(\S+)\s+(\d+)\s+src=(\w+)", line)
            if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == want:
                return int(m.group(3))
    return None


def _tiles_per_chunk(rn, dims) -> int:
    """Lattice tiles whose intermediates a plan holds at once, read back from
    the workspace size: each tile of a chunk adds 128 rows of bf16 z and
    scores and a 16-byte posterior record per row (and, with e4m3 scores,
    the rows' e4m3 z)."""
    import copy
    one = copy.copy(dims)
    one.tile_cells = 128
    per_tile = 128 * (2 * dims.H + 2 * dims.V + 16 + (dims.H if dims.dtype == rn.RNNT_BF16_E4M3
                                                        else 0))
    extra = rn.rnnt_workspace_bytes(dims) - rn.rnnt_workspace_bytes(one)
    return 1 + int(round(extra / per_tile))


def reduce_max(x: float, dist, device) -> float:
    """Max of a per-rank float over all ranks (the slowest rank sets the job time)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(cells_per_rank: int, world: int, ms: float) -> float:
    """Whole-job cells/s: every rank processes its own batch (weak scaling)."""
    return cells_per_rank * world / (ms / 1e3)


def run_gpu_bench(args):
    import numpy as np
    import torch

    import asr_tiled_tanh_gb300 as rn
    from asr_tiled_tanh_gb300 import shard, synthetic

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    rn.load(build_if_missing=True)

    wl = synthetic.WORKLOADS[args.workload]
    if args.batch > 0:  # the workload's shapes and distributions with another batch size
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}-B{args.batch}", B=args.batch)
    inp = synthetic.make(wl, seed=wl.seed + 1000 * rank)
    valid = inp.valid_cells()
    nominal = wl.nominal_cells
    e4m3 = args.scores == "e4m3"
    if args.budget_gb > 0:  # tile size from a memory budget for the library's buffers
        bdims = rn.make_dims(wl.B, wl.T, wl.U1, wl.HA, wl.HL, wl.H, wl.V, 0,
                             rn.RNNT_BF16_E4M3 if e4m3 else rn.binding.DTYPES[wl.dtype],
                             rn.RNNT_TILED, 0)
        args.tile_cells = rn.rnnt_tile_cells_for_budget(bdims, int(args.budget_gb * 1e9))
        if args.tile_cells <= 0:
            raise SystemExit(f"no tile size fits {args.budget_gb} GB")
    r = rn.Rnnt.for_inputs(inp, mode=args.mode, tile_cells=args.tile_cells, device=dev,
                           e4m3_scores=e4m3)
    d = {k: getattr(inp, k).to(dev) for k in ("hA", "hL", "WA", "WL", "bZ", "WO", "bO", "labels",
                                               "T_len", "U_len")}
    params = rn.make_params(d["WA"], d["WL"], d["bZ"], d["WO"], d["bO"])
    # parameter gradients in one flat buffer: with several ranks, one
    # all-reduce (sum) of it ends every step (data-parallel training)
    grad_flat, grads = shard.alloc_grads(wl.B, wl.T, wl.U1, wl.HA, wl.HL, wl.H, wl.V, device=dev)
    loss = torch.empty(wl.B, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(max(1, args.flush_mb) << 20, dtype=torch.uint8, device=dev)

    def step(s=stream, x=None):
        x = d if x is None else x  # the batch's device inputs
        if args.api == "step":  # rnnt_fwd_bwd: one call for the training step
            r.fwd_bwd(x["hA"], x["hL"], params, x["labels"], x["T_len"], x["U_len"], loss=loss,
                      grads=grads, stream=s)
        else:
            r.fwd(x["hA"], x["hL"], params, x["labels"], x["T_len"], x["U_len"], loss=loss,
                  stream=s)
            r.bwd(x["hA"], x["hL"], params, x["labels"], x["T_len"], x["U_len"], grads=grads,
                  stream=s)
        if dist is not None:
            with torch.cuda.stream(s):
                shard.allreduce_param_grads(grad_flat, dist)

    def captured(fn):
        """fn (which launches on the stream it is given) as a CUDA graph whose
        replay runs on the current stream."""
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            fn(cap)  # warm-up on the capture stream
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn(cap)
        torch.cuda.synchronize()
        return g

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    code, word = r.status()
    if code != 0:
        raise SystemExit(f"device status {code} word {word}")

    # A plan whose calls make no host synchronization (the whole lattice fits
    # one chunk of the tile buffers) is replayed as a CUDA graph of the step.
    use_graph = not args.eager and rn.rnnt_graph_capturable(r.dims) == 1 and dist is None
    graph = captured(step) if use_graph else None
    run = graph.replay if graph is not None else step

    def timed_region(fn, profile):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        if profile:
            rn.rnnt_profile_start(1 << 16)
        with ClockSampler(dev.index) as clk:
            t0 = time.perf_counter()
            for i in range(args.steps):
                if args.flush_mb > 0:
                    flush.fill_(i & 0xff)
                starts[i].record(stream)
                fn()
                ends[i].record(stream)
            clk.sample_now()
            torch.cuda.synchronize()
            wall = time.perf_counter() - t0
        prof = rn.rnnt_profile_stop() if profile else None
        if dist:
            dist.barrier()
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return sum(step_ms) / len(step_ms), clk, wall, prof, step_ms

    # --- timed region: device-resident inputs ---------------------------------
    torch.cuda.reset_peak_memory_stats(dev)
    ms, clk, wall, _, step_ms = timed_region(run, profile=False)
    peak_bytes = torch.cuda.max_memory_allocated(dev)
    ms_max = reduce_max(ms, dist, dev)
    value = job_value(nominal, world, ms_max)
    # what the timed steps ran (the peak measurement below builds another plan)
    timed_tile_cells = int(r.dims.tile_cells)
    timed_tiles_per_chunk = _tiles_per_chunk(rn, r.dims)
    execution = "CUDA graph of the step" if graph is not None else "eager"
    # --- the same steps again, eager, with every kernel bracketed by CUDA
    # events on its own stream: per-kernel times, shares and launch counts
    prof_ms, _, _, prof, _ = timed_region(step, profile=True)

    # --- the forward and the backward timed apart (eager, separate calls) ----
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        if args.flush_mb > 0:
            flush.fill_(i & 0xff)
        ev[i][0].record(stream)
        r.fwd(d["hA"], d["hL"], params, d["labels"], d["T_len"], d["U_len"], loss=loss)
        ev[i][1].record(stream)
        r.bwd(d["hA"], d["hL"], params, d["labels"], d["T_len"], d["U_len"], grads=grads)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    phases = {"api": "rnnt_fwd then rnnt_bwd, eager, L2 flushed before each step",
              "fwd_median": round(statistics.median(fwd_ms), 4),
              "bwd_median": round(statistics.median(bwd_ms), 4),
              "fwd_bwd_median": round(statistics.median(f + b for f, b in zip(fwd_ms, bwd_ms)), 4),
              "timed_step_median": round(statistics.median(step_ms), 4)}

    # --- e2e: host buffers through the C ABI ----------------------------------
    e2e_ms, h2d, d2h = None, 0, 0
    if not args.no_e2e:
        host_in = {k: getattr(inp, k).pin_memory() for k in ("hA", "hL", "labels", "T_len",
                                                              "U_len")}
        host_loss = torch.empty(wl.B, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = host_loss.numel() * 4

        def e2e_step(s=stream):
            with torch.cuda.stream(s):
                for k, v in host_in.items():
                    d[k].copy_(v, non_blocking=True)
                step(s)
                host_loss.copy_(loss, non_blocking=True)

        for _ in range(max(1, args.warmup // 2)):
            e2e_step()
        torch.cuda.synchronize()
        if use_graph:
            # one graph per step: batch in, step, losses out
            e2e_run = captured(e2e_step).replay
            es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            if dist:
                dist.barrier()
            for i in range(args.steps):
                flush.fill_(i & 0xff)
                es[i].record(stream)
                e2e_run()
                ee[i].record(stream)
            torch.cuda.synchronize()
            e2e_ms = sum(s.elapsed_time(e) for s, e in zip(es, ee)) / args.steps
            e2e_run = None
        else:
            # as a training loop feeds it: two device input buffers, the next
            # step's batch copied from pinned host memory on a copy stream
            # while the current step runs (every copy stays inside the timed
            # region; the step waits for its own batch)
            bufs = [{k: d[k] for k in host_in}, {k: torch.empty_like(d[k]) for k in host_in}]
            cs = torch.cuda.Stream(device=dev)
            copied = [torch.cuda.Event() for _ in range(2)]
            freed = [torch.cuda.Event() for _ in range(2)]

            def stage(i):
                j = i % 2
                if i >= 2:
                    cs.wait_event(freed[j])  # the step that read buffer j is done
                with torch.cuda.stream(cs):
                    for k, v in host_in.items():
                        bufs[j][k].copy_(v, non_blocking=True)
                    copied[j].record(cs)

            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            if dist:
                dist.barrier()
            torch.cuda.synchronize()
            t0.record(stream)
            cs.wait_event(t0)
            stage(0)
            for i in range(args.steps):
                if i + 1 < args.steps:
                    stage(i + 1)
                flush.fill_(i & 0xff)
                stream.wait_event(copied[i % 2])
                step(stream, bufs[i % 2])
                freed[i % 2].record(stream)
                host_loss.copy_(loss, non_blocking=True)
            t1.record(stream)
            torch.cuda.synchronize()
            e2e_ms = t0.elapsed_time(t1) / args.steps
            bufs = None
        e2e_ms = reduce_max(e2e_ms, dist, dev)
        assert np.isfinite(host_loss.numpy()).all()

    # --- peak HBM at a second tile size -------------------------------------------
    # Tiled mode holds the large intermediates only for the tiles of one chunk,
    # so the peak should move with the tile buffers and not with B*T*U*V.  The
    # first plan's buffers are freed, a plan with a quarter of its tiles per
    # chunk (whole waves of SMs) runs one step, and both peaks are reported
    # with their tiles per chunk.
    tiles_first = timed_tiles_per_chunk
    peak_by_tiles = {str(tiles_first): round(peak_bytes / 1e9, 4)}
    peak_tc = args.peak_tile_cells
    if peak_tc < 0 and args.mode == "tiled":
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        peak_tc = max(nsm, (tiles_first // 4) // nsm * nsm) * 128
    if peak_tc > 0 and args.mode == "tiled" and peak_tc < tiles_first * 128:
        graph = run = None
        r.saved = r.ws = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        r = rn.Rnnt.for_inputs(inp, mode=args.mode, tile_cells=peak_tc, device=dev,
                               e4m3_scores=e4m3)
        step()
        torch.cuda.synchronize()
        code, word = r.status()
        if code != 0:
            raise SystemExit(f"device status {code} word {word} (second tile size)")
        peak_by_tiles[str(_tiles_per_chunk(rn, r.dims))] = \
            round(torch.cuda.max_memory_allocated(dev) / 1e9, 4)

    # --- the same workload with the score products on e4m3 tensor cores --------
    # A secondary line (`value` is the bf16 path's): RNNT_BF16_E4M3, timed like
    # the main steps on a plan of its own, so that every default run also
    # records the reduced-precision option on the same box.
    e4m3_leg = None
    if args.e4m3_leg and not e4m3 and wl.dtype == "bf16" and dist is None:
        graph = run = None
        r.saved = r.ws = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        r = rn.Rnnt.for_inputs(inp, mode=args.mode, tile_cells=args.tile_cells, device=dev,
                               e4m3_scores=True)
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        code, word = r.status()
        if code != 0:
            raise SystemExit(f"device status {code} word {word} (e4m3 scores)")
        g8 = captured(step) if (not args.eager and rn.rnnt_graph_capturable(r.dims) == 1) \
            else None
        ms8, clk8, _, _, _ = timed_region(g8.replay if g8 is not None else step, profile=False)
        g8 = None
        ms8 = reduce_max(ms8, dist, dev)
        e4m3_leg = {"dtype": "bf16+e4m3", "ms_per_step": round(ms8, 4),
                    "value": round(job_value(nominal, world, ms8), 1), "unit": UNIT,
                    "scores": "W^O per 256-row block with power-of-two scales, z as e4m3(2^8 z); "
                              "dz, dW^O and the rest bf16",
                    "clocks": clk8.summary()}

    # --- roofline of the dominant kernel ----------------------------------------
    hbm_peak, tf_burst, tf_sust, peak_src = _peaks()
    # the burst figure for a short timed region, the power-capped sustained
    # one once the timed region runs for a second or more
    peak_kind = "sustained" if ms_max * args.steps >= 1000.0 else "burst"
    peak_tf = tf_sust if peak_kind == "sustained" else tf_burst
    launches = sum(c for _, c in prof.values())
    # the ncu summaries key their traffic figures by workload (and mode)
    traffic_key = wl.name if args.mode == "tiled" else f"{wl.name}-untiled"
    if e4m3:
        traffic_key += "-e4m3"
    top = max(prof.items(), key=lambda kv: kv[1][0]) if prof else ("none", (0.0, 1))
    top_name, (top_ms, top_n) = top
    H, V = wl.H, wl.V
    roof = None
    if top_name in KERNEL_FLOPS_PER_CELL_HV:
        flops_per_launch = KERNEL_FLOPS_PER_CELL_HV[top_name] * H * V * valid \
            / max(1, top_n // args.steps)
        ach = flops_per_launch / (top_ms / top_n / 1e3) / 1e12
        peak, src = peak_tf, f"{peak_src} bf16 {peak_kind}"
        if e4m3 and top_name in E4M3_KERNELS:
            # a contraction takes the peak of its own dtype: the measured bf16
            # figure times the nominal dense e4m3 / bf16 ratio (4.5 / 2.25)
            peak, src = 2.0 * peak_tf, f"{src} x 2 (nominal dense e4m3/bf16 ratio)"
        roof = {"kernel": top_name, "bound": "tensor", "achieved": round(ach, 2),
                "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                "traffic": recorded_traffic(top_name, traffic_key),
                "peak_source": src,
                "flops_per_launch": flops_per_launch, "launches": top_n,
                "avg_launch_ms": top_ms / top_n}
    elif top_name in KERNEL_BYTES_PER_CELL:
        bytes_per_launch = KERNEL_BYTES_PER_CELL[top_name](V) * valid / max(1, top_n // args.steps)
        ach = bytes_per_launch / (top_ms / top_n / 1e3) / 1e9
        roof = {"kernel": top_name, "bound": "hbm", "achieved": round(ach, 1),
                "peak": hbm_peak, "unit": "GB/s", "frac": round(ach / hbm_peak, 4),
                "traffic": recorded_traffic(top_name, traffic_key),
                "peak_source": f"{peak_src} copy bandwidth",
                "bytes_per_launch": bytes_per_launch, "launches": top_n,
                "avg_launch_ms": top_ms / top_n}
    else:
        roof = {"kernel": top_name, "bound": "alu", "achieved": None, "peak": None,
                "unit": "TFLOP/s", "frac": None, "traffic": None,
                "note": "fp32 FFMA kernels; no tensor-core phase"}
    shares = {k: round(v[0] / sum(x[0] for x in prof.values()), 4) for k, v in
              sorted(prof.items(), key=lambda kv: -kv[1][0])}

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16+e4m3" if e4m3 else "bf16") if wl.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": f"{wl.name}: B={wl.B} T={wl.T} U={wl.U} HA=HL=H={wl.H} "
                               f"V={wl.V} {wl.dtype}", "B": wl.B, "T": wl.T, "U": wl.U,
                   "H": wl.H, "V": wl.V, "tile_cells": timed_tile_cells,
                   "tiles_per_chunk": timed_tiles_per_chunk,
                   "nominal_cells": nominal, "valid_cells": valid,
                   "l2": "flushed (256 MiB write) before each timed step",
                   "execution": execution,
                   "mode": args.mode,
                   "scores": ("e4m3 (W^O per 256-row block, power-of-two scales; z as "
                              "e4m3(2^8 z)); dz, dW^O and the rest bf16" if e4m3 else "bf16"),
                   "api": "rnnt_fwd_bwd" if args.api == "step" else "rnnt_fwd + rnnt_bwd",
                   "parallelism": f"dp{world}",
                   "collective": ("one all-reduce (sum, NCCL) of the parameter gradients per "
                                  "step" if world > 1 else "none")},
        "valid_cells_per_s": round(valid * world / (ms_max / 1e3), 1),
        "peak_hbm_gb": round(peak_bytes / 1e9, 4),
        "peak_hbm_gb_by_tiles_per_chunk": peak_by_tiles,
        "bf16_peak_frac_6HV": round(6 * H * V * valid / (ms_max / 1e3) / 1e12 / peak_tf, 4),
        # executed products: the tiled backward recomputes the scores (8HV per
        # valid position); the untiled one keeps them (6HV)
        "bf16_peak_frac_executed": round((8 if args.mode == "tiled" else 6) * H * V * valid
                                         / (ms_max / 1e3) / 1e12 / peak_tf, 4),
        "ms_by_phase": phases,
        "e2e": None if e2e_ms is None else {
            "value": round(job_value(nominal, world, e2e_ms), 1), "unit": UNIT,
            "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "inputs": ("copied inside each replayed step graph" if use_graph else
                       "next step's batch copied on a second stream during the current "
                       "step (two device input buffers)")},
        "gpu_launches": int(launches),
        "roofline": roof,
        "kernel_shares": shares,
        "kernel_ms_per_step": {k: round(v[0] / args.steps, 5) for k, v in
                               sorted(prof.items(), key=lambda kv: -kv[1][0])},
        "profiled_ms_per_step": round(prof_ms, 4),
        "e4m3_scores": e4m3_leg,
        "clocks": clk.summary(),
        "wall_s_timed": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def _by_size(inp):
    """Sample indices of a batch from the smallest lattice to the largest."""
    cells = (inp.T_len.long() * (inp.U_len.long() + 1)).tolist()
    return sorted(range(len(cells)), key=lambda b: (cells[b], b))


def _oracle_sample(inp, idx):
    """The oracle, fwd+bwd in fp64, on the samples `idx` of the batch:
    (seconds, the sub-batch)."""
    import oracle
    sub = inp.subset(list(idx))
    f = lambda t: t.double().numpy()
    t0 = time.perf_counter()
    oracle.rnnt(f(sub.hA), f(sub.hL), f(sub.WA), f(sub.WL), f(sub.bZ), f(sub.WO), f(sub.bO),
                sub.labels.numpy(), sub.T_len.numpy(), sub.U_len.numpy())
    return time.perf_counter() - t0, sub


def nominal_equivalent(valid_cells_per_s: float, inp) -> float:
    """A rate over valid lattice positions expressed in the metric's unit
    (nominal cells B*T*(U+1) per second of the whole batch): the oracle's cost
    is per valid position, so a sample's valid-position rate is scaled by the
    batch's nominal / valid ratio."""
    return valid_cells_per_s * inp.wl.nominal_cells / max(1, inp.valid_cells())


def cpu_baseline(inp, budget_s):
    """The oracle, as it stands, on a bounded sample of the same workload: the
    smallest lattices of the batch first, as many as fit the time budget."""
    import oracle
    oracle.build()
    order = _by_size(inp)
    n = 1
    dt, sub = _oracle_sample(inp, order[:1])
    if dt < budget_s / 3 and inp.wl.B > 1:
        n = max(1, min(inp.wl.B, int(budget_s / max(dt, 1e-3))))
        dt, sub = _oracle_sample(inp, order[:n])
    valid = sub.valid_cells()
    return {"value": round(nominal_equivalent(valid / dt, inp), 2), "unit": UNIT,
            "cores": oracle.num_threads(), "kind": "oracle", "seconds": round(dt, 3),
            "valid_cells_per_s": round(valid / dt, 2),
            "sample": f"the {n} smallest lattice(s) of the workload's batch, fwd+bwd, fp64 "
                      f"({valid} valid positions in {dt:.1f} s); value = that valid-position "
                      f"rate x the batch's nominal/valid ratio "
                      f"({inp.wl.nominal_cells}/{inp.valid_cells()})"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from asr_tiled_tanh_gb300 import synthetic
    import oracle
    oracle.build()
    wl = synthetic.WORKLOADS[args.workload]
    inp = synthetic.make(wl)
    # one step = the oracle on a bounded sample of the workload: the batch's
    # smallest lattice (the full batch would take the oracle hours)
    idx = _by_size(inp)[:1]
    for _ in range(min(args.warmup, 1)):
        _oracle_sample(inp, idx)
    times = []
    for _ in range(args.steps):
        dt, sub = _oracle_sample(inp, idx)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    valid = sub.valid_cells()
    value = nominal_equivalent(valid / (ms / 1e3), inp)
    sample = (f"sample {idx[0]} of the workload's batch (its smallest lattice: T_b="
              f"{int(sub.T_len[0])}, U_b={int(sub.U_len[0])}, {valid} valid positions), fwd+bwd, "
              f"fp64, per step; value = its valid-position rate x the batch's nominal/valid "
              f"ratio ({wl.nominal_cells}/{inp.valid_cells()})")
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
           "n_gpus": args.gpus, "device": "host cores (the oracle runs on no GPU)",
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": f"{wl.name}: B={wl.B} T={wl.T} U={wl.U} HA=HL=H={wl.H} "
                                  f"V={wl.V} {wl.dtype}", "B": wl.B, "T": wl.T, "U": wl.U,
                      "H": wl.H, "V": wl.V, "sample": sample},
           "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "kind": "oracle",
                            "cores": oracle.num_threads(), "sample": sample},
           "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="audio40",
                    help="synthetic workload (asr_tiled_tanh_gb300/synthetic.py); the default "
                         "is the 40 s, batch-1024 configuration")
    ap.add_argument("--tile-cells", type=int, default=0)
    ap.add_argument("--budget-gb", type=float, default=0.0,
                    help="choose tile_cells so that the library's saved + workspace buffers "
                         "fit this many GB (rnnt_tile_cells_for_budget)")
    ap.add_argument("--peak-tile-cells", type=int, default=-1,
                    help="after the timed steps, peak HBM of one step at this second tile "
                         "size (-1: a quarter of the first plan's tile buffers; 0: skip)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush-mb", type=int, default=256,
                    help="L2 flush buffer written before each timed step (0: none; profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling)")
    ap.add_argument("--batch", type=int, default=0,
                    help="samples per batch (0: the workload's own B); for profiling on "
                         "smaller cases of a workload's shapes")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step eagerly instead of replaying a CUDA graph")
    ap.add_argument("--api", default="step", choices=["step", "separate"],
                    help="step: one rnnt_fwd_bwd call per step; separate: rnnt_fwd + rnnt_bwd")
    ap.add_argument("--scores", default="bf16", choices=["bf16", "e4m3"],
                    help="e4m3: the two score products on e4m3 tensor cores (RNNT_BF16_E4M3)")
    ap.add_argument("--no-e4m3-leg", dest="e4m3_leg", action="store_false",
                    help="skip the secondary timing of a bf16 workload with e4m3 scores "
                         "(`e4m3_scores` in the JSON line)")
    ap.add_argument("--mode", default="tiled", choices=["tiled", "untiled"],
                    help="untiled keeps z and the scores from the forward (no recompute)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not started by a launcher: start one process per GPU here
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
        raise SystemExit(subprocess.call(cmd))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu_bench(args)


if __name__ == "__main__":
    main()

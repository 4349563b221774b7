"""Benchmark: layout_copy GB/s (bytes read + written) on GB300.

One step = one pass of the relayout suite, each workload one layout_copy
through the C ABI:

  C2  fp32 4096x4096 column-major -> row-major             (STAGED)
  C3  bf16 8192x8192 -> 64x64 tiles, Swizzle<3,4,3> inside (VEC 16 B)
  C4  fp64 2^20 padded 8x8 tiles gathered into TV order    (STAGED)
  C5a fp16 NHWC (64,56,56,256) -> NCHW                     (STAGED)
  C5b fp16 (2,16384,128) head-major -> stride-2 interleave (ZIP)

value = algorithmic bytes (every element read and written once; C4's
source also counts its pad slots, which share DRAM sectors with the data)
over the CUDA-event time of the steps, on the launching stream.  The five
buffer pairs (1.87 GB per step) are each reused only after > 1.6 GB of other
traffic, larger than the 126 MiB L2, so no explicit flush is done.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the whole suite on its own GPU (weak
scaling, no collective on the data path); rank 0 prints the line with the
max-over-ranks time.  ``--impl reference`` times the CPU oracle instead.
"""

from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import BENCH_SUITE, WORKLOADS, seeded_bytes  # noqa: E402

METRIC = ("layout_copy GB/s (read+write) and % of GB300 HBM peak; "
          "bit-exact vs CPU oracle")
UNIT = "GB/s"
# algorithmic bytes per copy (read + written; C4 reads 72 source slots per
# 64-element tile)
ALGO_BYTES = {"C2": 134_217_728, "C3": 268_435_456, "C4": 1_140_850_688,
              "C5a": 205_520_896, "C5b": 16_777_216}
DOMINANT = "C4"          # largest share of the step: lm_bulk_kernel<8>

# The thread-value tile copy (lm_tv_copy) on full-size workloads: shared
# tile layout, thread layouts of the load and store phases, and the tiler
# that zipped_divide applies to both sides first (None: the workload's
# layouts are tiled already).  Reported beside the suite, not part of the
# headline.
TV_CONFIGS = {
    # bf16 64x64 tiles, 16-byte vectors along the contiguous columns in both
    # phases, 128-byte XOR swizzle on the shared rows
    "C3": ("Sw<3,3,6> o (64,64):(64,1)", "(32,8):(8,1)", "(32,8):(8,1)",
           None),
    # fp32 64x64 transposes: 4-byte accesses in both phases, a 5-bit XOR so
    # a warp reading a shared row or column touches 32 banks
    "C2": ("Sw<5,0,6> o (64,64):(1,64)", "(32,8):(1,32)", "(8,32):(32,1)",
           (64, 64)),
    # the same with 16-byte loads; the store phase then conflicts 4 ways
    "C2v": ("Sw<3,2,6> o (64,64):(1,64)", "(16,16):(1,16)", "(8,32):(32,1)",
            (64, 64)),
    # the conflict-free tile with the planner's tuned stripmined thread
    # layouts (no thread layout given)
    "C2t": ("Sw<5,0,6> o (64,64):(1,64)", None, None, (64, 64)),
}
FALLBACK_HBM_GBS = 6800.0
E2E_ROUNDS = 3


def peaks() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 50 ms) of the GPU under test; only samples
    stamped inside the sampled window count.  The window is the suite
    running without a break for SOAK_S seconds before and after the timed
    steps, which sit inside it (the timed steps alone last milliseconds,
    shorter than the sampling interval)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
               "sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.window = (0.0, float("inf"))

    def __enter__(self):
        if not self.gpu:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        import datetime
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(
                    parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        reasons = sorted({name for r in use for name, flag in
                          zip(self.REASONS, r[3]) if flag.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": reasons,
                "samples": len(use), "in_timed_window": bool(inside)}


def gpu_smi_id(local: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        first = vis.split(",")[local] if vis else str(local)
        return first.strip()


# --------------------------------------------------------------------------
# the suite on the GPU
# --------------------------------------------------------------------------

class Suite:
    def __init__(self, device, names=BENCH_SUITE):
        import torch
        import layout_driven_movement_gb300 as lm
        self.torch, self.lm = torch, lm
        self.items = []
        for name in names:
            w = WORKLOADS[name]
            S, D = lm.build_layout(w.src), lm.build_layout(w.dst)
            plan = lm.Plan(S, D, w.elem_bytes)
            # the source buffer holds whole 16-byte chunks (C4: 2^20 whole
            # 72-element tiles; its last pad slot lies past the cosize)
            n_src = -(-(S.cosize * w.elem_bytes) // 16) * 16 // w.elem_bytes
            host = seeded_bytes(w.values, w.dtype, n_src, w.seed)
            src = torch.from_numpy(host).to(device)
            dst = torch.empty(D.cosize * w.elem_bytes, dtype=torch.uint8,
                              device=device)
            self.items.append(dict(name=name, w=w, plan=plan, src=src,
                                   dst=dst, host=host, S=S, D=D,
                                   bytes=ALGO_BYTES[name]))
        self.bytes_per_step = sum(it["bytes"] for it in self.items)
        self.launches_per_step = sum(it["plan"].launches for it in self.items)

    def step(self, events=None):
        lm = self.lm
        for k, it in enumerate(self.items):
            if events is not None:
                events[k][0].record()
            lm.layout_copy(it["plan"], it["src"], it["dst"])
            if events is not None:
                events[k][1].record()


def run_native(args) -> dict | None:
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        import __graft_entry__ as g
        g.build()
    if world > 1:
        dist.barrier()
    import layout_driven_movement_gb300 as lm
    lm.lib()
    names = tuple(args.workloads.split(",")) if args.workloads else BENCH_SUITE
    suite = Suite(device, names)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        suite.step()
    torch.cuda.synchronize()

    n = len(suite.items)
    ev0, ev1 = (torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True))
    # steps of uninterrupted load around the timed steps, so the clock
    # sampler sees the GPU in the state the timed steps run in
    soak = 0 if args.quick else soak_steps(suite, torch)
    with ClockSampler(gpu_smi_id(local) if not args.quick else "") as clk:
        if not args.quick:
            time.sleep(0.5)         # let the sampler start
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start = time.time()
        for _ in range(soak):
            suite.step()
        # the headline region: K steps back to back, events only at its ends,
        # so consecutive copies overlap launch and tail (programmatic
        # dependent launch keeps their stream order)
        ev0.record()
        for _ in range(args.steps):
            suite.step()
        ev1.record()
        for _ in range(soak):
            suite.step()
        torch.cuda.synchronize()
        clk.window = (t_start, time.time())
        if world > 1:
            dist.barrier()
    total_ms = ev0.elapsed_time(ev1)
    wall = total_ms * 1e-3
    # per-copy breakdown: a second timed pass with events around every copy
    k2 = min(args.steps, 1000)
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(n)] for _ in range(k2)]
    torch.cuda.synchronize()
    for s in range(k2):
        suite.step(events[s])
    torch.cuda.synchronize()
    per = {it["name"]: [] for it in suite.items}
    for s in range(k2):
        for k, it in enumerate(suite.items):
            per[it["name"]].append(events[s][k][0].elapsed_time(events[s][k][1]))
    if world > 1:
        t = torch.tensor([total_ms, wall], dtype=torch.float64)
        gathered = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(gathered, t)
        total_ms = max(float(g[0]) for g in gathered)
        wall = max(float(g[1]) for g in gathered)
    value = suite.bytes_per_step * args.steps * world / (total_ms * 1e-3) / 1e9
    # the bulk-copy kernels bound their waits on the device; a wait that gave
    # up would leave part of a destination unwritten, so no number stands
    if lm.device_status() != 0:
        raise RuntimeError("a copy kernel gave up a bounded wait "
                           "(LM_E_TIMEOUT): the run is invalid")

    peak, peak_kind = peaks()
    iso = isolated_times(suite, torch) if not args.quick else {}
    mcp = memcpy_times(suite, torch, k2) if not args.quick else {}
    per_cfg = {}
    for it in suite.items:
        ms = statistics.median(per[it["name"]])
        gbs = it["bytes"] / (ms * 1e-3) / 1e9
        pieces = it["plan"].describe()["pieces"]
        per_cfg[it["name"]] = {
            "path": "+".join(p["path"] for p in pieces),
            "kernel": kernel_name(it["plan"], it["w"].elem_bytes),
            # shared-memory wavefronts per launch predicted by the planner's
            # bank-conflict simulation ([predicted, conflict-free minimum]):
            # the store side's shared loads, and the 16-byte tile writes
            # (cp.async, or the bulk copy engine when "bulk" is set)
            "smem_read_wavefronts": staged_sum(
                pieces, "bank_read_wavefronts", "bank_read_wavefronts_ideal"),
            "smem_write_wavefronts": staged_sum(
                pieces, "bank_wavefronts", "bank_wavefronts_ideal",
                minus=("bank_read_wavefronts", "bank_read_wavefronts_ideal")),
            "bytes": it["bytes"], "median_us": round(ms * 1e3, 2),
            "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
        if it["name"] in iso:
            ims = iso[it["name"]]
            igbs = it["bytes"] / (ims * 1e-3) / 1e9
            per_cfg[it["name"]].update({
                "isolated_us": round(ims * 1e3, 2),
                "isolated_frac_of_peak": round(igbs / peak, 4)})
        if it["name"] in mcp:
            nb, m_suite, m_alone = mcp[it["name"]]
            per_cfg[it["name"]]["memcpy"] = {
                "bytes": nb, "median_us": round(m_suite * 1e3, 2),
                "frac_of_peak": round(nb / (m_suite * 1e-3) / 1e9 / peak, 4),
                "isolated_us": round(m_alone * 1e3, 2),
                "isolated_frac_of_peak": round(
                    nb / (m_alone * 1e-3) / 1e9 / peak, 4)}
    dom_name = DOMINANT if DOMINANT in per else suite.items[0]["name"]
    dom_item = next(it for it in suite.items if it["name"] == dom_name)
    dom_kernel = kernel_name(dom_item["plan"], dom_item["w"].elem_bytes)
    dom = per[dom_name]
    dom_ms = sum(dom) / len(dom)
    achieved = ALGO_BYTES[dom_name] / (dom_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": measured_traffic(dom_kernel),
                "kernel": dom_kernel + " (" + dom_name + ")",
                "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s"}
    # end to end: every rank at once, the slowest rank's time
    e2e = None
    if not args.quick:
        if world > 1:
            dist.barrier()
        e2e = measure_e2e(suite, args, torch, shards=args.e2e_shards)
        if world > 1:
            t = torch.tensor([e2e["ms"]], dtype=torch.float64)
            gathered = [torch.zeros_like(t) for _ in range(world)]
            dist.all_gather(gathered, t)
            e2e["ms"] = max(float(g[0]) for g in gathered)
        e2e["value"] = round(suite.bytes_per_step * e2e["steps"] * world /
                             (e2e["ms"] * 1e-3) / 1e9, 1)
        del e2e["ms"]
    if rank != 0:
        return None

    ceiling = measure_d2d(suite, torch) if not args.quick else None
    other = measure_eval_and_generic(suite, torch, peak) if not args.quick else {}
    tv = measure_tv(suite, args, torch, peak) if not args.quick else {}
    xch = measure_exchange(suite, args, torch, peak) if not args.quick else {}
    cpu = cpu_baseline(suite) if world == 1 and not args.quick else None
    clocks = clk.summary()
    if soak:
        clocks["window"] = (f"the suite without a break: {soak} steps "
                            "before and after the timed steps, which lie "
                            "inside the sampled window")
        clocks["window_s"] = round(clk.window[1] - clk.window[0], 3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": "synthetic (seeded numpy PCG64, shapes and "
        "value distributions of the five relayouts)",
        "config": {
            "workload": "relayout suite " + "+".join(names) +
                        ", one layout_copy each per step",
            "bytes_per_step": suite.bytes_per_step,
            "element_types": "fp32, bf16, fp64, fp16, fp16 (moved as raw bytes)",
            "l2": "no flush: 1.87 GB/step over five buffer pairs, each reused "
                  "after >1.6 GB of other traffic (L2 126 MiB)",
            "wall_s_timed": round(wall, 4),
            "breakdown": "per_config: a second pass of " + str(k2) +
                         " steps with CUDA events around every copy; "
                         "isolated_*: each copy alone after a read flush of "
                         "L2; memcpy: a cudaMemcpyAsync of the copy's bytes "
                         "in its slot of the suite and alone",
            "per_config": per_cfg,
            "d2d_copy_ceiling_gbs": ceiling,
            "other_kernels": other,
            "tv_copy": tv,
            "exchange": xch,
        },
        "clocks": clocks,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": suite.launches_per_step * args.steps,
    }
    return line


SOAK_S = 0.6


def soak_steps(suite, torch) -> int:
    """Steps that keep the GPU busy for about SOAK_S seconds (from the time
    of a few steps)."""
    e0, e1 = (torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True))
    e0.record()
    for _ in range(10):
        suite.step()
    e1.record()
    torch.cuda.synchronize()
    per = max(e0.elapsed_time(e1) / 10, 1e-3)
    return int(SOAK_S * 1e3 / per) + 1


def staged_sum(pieces, key, ideal_key, minus=None):
    """A per-tile planner figure summed over the STAGED pieces' tiles."""
    got = [0, 0]
    for p in pieces:
        if p["path"] != "STAGED":
            continue
        a, b = p[key], p[ideal_key]
        if minus:
            a, b = a - p[minus[0]], b - p[minus[1]]
        got[0] += a * p["n_tiles"]
        got[1] += b * p["n_tiles"]
    return got if any(p["path"] == "STAGED" for p in pieces) else None


def kernel_name(plan, eb: int) -> str:
    """The CUDA kernel a one-piece plan launches, as ncu names it."""
    pc = plan.describe()["pieces"][0]
    if pc["path"] == "STAGED":
        store = (f"XposeStore<{eb}, {pc['rows']}>" if pc["store"] == "transpose"
                 else f"GatherStore<{eb}>")
        if pc["bulk"]:
            # ncu prints the bool template argument as 0 / 1
            tma = 1 if pc.get("tma") else 0
            return f"lm_bulk_kernel<{eb}, {store}, {pc['stages']}, {tma}>"
        return f"lm_staged_kernel<{eb}, {store}, {pc['stages']}>"
    if pc["path"] == "VEC":
        return f"lm_vec_tiled_kernel<{pc['vec_bytes']}, 4>"
    if pc["path"] == "ZIP":
        u = 2 if os.environ.get("LM_ZIP_UNROLL", "1").startswith("2") else 1
        return f"lm_zip_kernel<{eb}, {pc['rows']}, {u}>"
    return f"lm_generic_kernel<{eb}>"


def measured_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None if absent or taken on different kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)[kernel]
        src = os.path.join(ROOT, "layout_driven_movement_gb300", "csrc",
                           "lm_kernels.cu")
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if rec.get("kernel_source_sha") != sha:
            return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


def isolated_times(suite, torch, runs=20) -> dict:
    """Each copy alone: L2 flushed before every run by reading a 512 MiB
    buffer (which writes back the previous copy's dirty lines and leaves
    only clean ones), the copy timed by events around it, median over
    `runs` (ms) -- the kernel without its neighbours' write-backs and launch
    overlap."""
    dev = suite.items[0]["src"].device
    flush = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    lm = suite.lm
    out = {}
    for it in suite.items:
        times = []
        for r in range(runs + 3):
            flush.max()
            e0, e1 = (torch.cuda.Event(enable_timing=True),
                      torch.cuda.Event(enable_timing=True))
            e0.record()
            lm.layout_copy(it["plan"], it["src"], it["dst"])
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                times.append(e0.elapsed_time(e1))
        out[it["name"]] = statistics.median(times)
    del flush
    return out


def memcpy_times(suite, torch, steps, runs=20) -> dict:
    """The same-run reference for the per-copy figures: a device-to-device
    memcpy (torch's copy_, cudaMemcpyAsync) from each copy's source buffer
    into its destination buffer of as many bytes as the copy moves -- half
    read, half written, at most either buffer.  Timed in the copy's slot of
    the suite (the suite with every copy replaced by its memcpy, events
    around each, median over `steps`, so each memcpy also writes back its
    predecessors' dirty lines) and alone after a read flush of L2 (as
    isolated_times).  Returns {name: (bytes, suite ms, isolated ms)}."""
    pairs = []
    for it in suite.items:
        src, dst = it["src"].view(torch.uint8), it["dst"].view(torch.uint8)
        n = min(it["bytes"] // 2, src.numel(), dst.numel())
        pairs.append((it["name"], src[:n], dst[:n]))
    for _ in range(3):
        for _, s, d in pairs:
            d.copy_(s)
    ev = [[(torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in pairs]
          for _ in range(steps)]
    torch.cuda.synchronize()
    for row in ev:
        for (e0, e1), (_, s, d) in zip(row, pairs):
            e0.record()
            d.copy_(s)
            e1.record()
    torch.cuda.synchronize()
    flush = torch.ones(512 << 20, dtype=torch.uint8, device=pairs[0][1].device)
    out = {}
    for k, (name, s, d) in enumerate(pairs):
        in_suite = statistics.median(row[k][0].elapsed_time(row[k][1])
                                     for row in ev)
        alone = _timed(torch, lambda: d.copy_(s), runs, flush)
        out[name] = (2 * s.numel(), in_suite, alone)
    del flush
    return out


def _timed(torch, fn, runs=20, flush=None):
    """Median event time (ms) of fn, L2 flushed by a read before each run."""
    times = []
    for r in range(runs + 3):
        if flush is not None:
            flush.max()
        e0, e1 = (torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True))
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        if r >= 3:
            times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def measure_eval_and_generic(suite, torch, peak) -> dict:
    """The kernels the suite does not time.  layout_eval: the offset table
    of the padded TV source layout (67 M entries, int64: 537 MB written),
    beside a write-only fill of the same bytes (the write ceiling).
    GENERIC: a 6000x7000 fp32 relayout whose two layouts have no common
    refinement, one element per thread with a full decomposition on each
    side; and the 6000x7000 pair that refines once a side is coalesced."""
    lm = suite.lm
    dev = suite.items[0]["src"].device
    flush = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    out = {}
    it = next((i for i in suite.items if i["name"] == "C4"), None)
    if it is not None:
        L = it["S"]
        table = torch.empty(L.size, dtype=torch.int64, device=dev)
        ms = _timed(torch, lambda: lm.layout_eval_device(L, table),
                    flush=flush)
        gbs = L.size * 8 / (ms * 1e-3) / 1e9
        fill_ms = _timed(torch, lambda: table.fill_(7), flush=flush)
        fill_gbs = L.size * 8 / (fill_ms * 1e-3) / 1e9
        out["layout_eval"] = {
            "workload": "offset table of the padded TV source layout, "
                        f"{L.size} int64 entries", "median_us": round(ms * 1e3, 2),
            "gbs_written": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "fill_ceiling_gbs": round(fill_gbs, 1),
            "frac_of_fill": round(gbs / fill_gbs, 4)}
        del table
    S = lm.Layout.parse("(6000,7000):(7000,1)")
    pairs = {
        # 6000 and 7000 do not nest and the padded destination does not
        # coalesce: no common refinement, one element per thread
        "generic": ("(7000,6000):(1,7001)",
                    "6000x7000 fp32 into a padded (7000,6000):(1,7001) "
                    "destination: no common refinement"),
        # the same matrix against (7000,6000):(1,7000), the single run
        # 42000000:1, refines into a transpose
        "coalesced_transpose": ("(7000,6000):(1,7000)",
                                "6000x7000 fp32 against (7000,6000):(1,7000)"
                                ", refined once the destination is seen "
                                "as one run: a transpose"),
    }
    for key, (d_txt, what) in pairs.items():
        D = lm.Layout.parse(d_txt)
        plan = lm.Plan(S, D, 4)
        a = torch.empty(S.cosize * 4, dtype=torch.uint8, device=dev)
        b = torch.empty(D.cosize * 4, dtype=torch.uint8, device=dev)
        ms = _timed(torch, lambda: lm.layout_copy(plan, a, b), flush=flush)
        gbs = 2 * S.size * 4 / (ms * 1e-3) / 1e9
        out[key] = {
            "workload": what,
            "path": "+".join(p["path"] for p in plan.describe()["pieces"]),
            "median_us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4)}
        del a, b
    del flush
    return out


def measure_d2d(suite, torch) -> float:
    """The practical ceiling on this GPU now: a plain device-to-device copy
    (cudaMemcpyAsync through torch) moving the suite's bytes per step --
    half of them read, half written -- timed like the suite, median of 30."""
    n = suite.bytes_per_step // 2
    a = torch.empty(n, dtype=torch.uint8, device=suite.items[0]["src"].device)
    b = torch.empty_like(a)
    for _ in range(3):
        b.copy_(a)
    times = []
    for _ in range(30):
        e0, e1 = (torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True))
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    del a, b
    return round(2 * n / (ms * 1e-3) / 1e9, 1)


def measure_tv(suite, args, torch, peak) -> dict:
    """Time lm_tv_copy on the suite's full-size buffers (TV_CONFIGS), the
    copies of one pass back to back with events around each (each then
    also writes back its predecessor's dirty lines), and each alone after a
    read flush of L2 (`isolated_us`)."""
    lm = suite.lm
    items = {it["name"]: it for it in suite.items}
    runs = []
    for key, (smem, tl, ts, tiler) in TV_CONFIGS.items():
        it = items.get(key[:2])
        if it is None:
            continue
        S, D = it["S"], it["D"]
        if tiler:
            S, D = S.zipped_divide(list(tiler)), D.zipped_divide(list(tiler))
        plan = lm.TVPlan(S, lm.Layout.parse(smem), D,
                         lm.Layout.parse(tl) if tl else None,
                         lm.Layout.parse(ts) if ts else None,
                         it["w"].elem_bytes)
        runs.append((key, it, plan))
    if not runs:
        return {}
    passes = min(args.steps, 300)
    for _ in range(3):
        for _, it, plan in runs:
            lm.tv_copy(plan, it["src"], it["dst"])
    ev = [[(torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in runs]
          for _ in range(passes)]
    torch.cuda.synchronize()
    for r in range(passes):
        for k, (_, it, plan) in enumerate(runs):
            ev[r][k][0].record()
            lm.tv_copy(plan, it["src"], it["dst"])
            ev[r][k][1].record()
    torch.cuda.synchronize()
    # each copy alone as well: L2 flushed by a read before each of 20 runs
    flush = torch.ones(512 << 20, dtype=torch.uint8,
                       device=suite.items[0]["src"].device)
    iso = {key: _timed(torch, lambda it=it, plan=plan:
                       lm.tv_copy(plan, it["src"], it["dst"]), flush=flush)
           for key, it, plan in runs}
    del flush
    out = {}
    for k, (key, it, plan) in enumerate(runs):
        ms = statistics.median(ev[r][k][0].elapsed_time(ev[r][k][1])
                               for r in range(passes))
        gbs = it["bytes"] / (ms * 1e-3) / 1e9
        igbs = it["bytes"] / (iso[key] * 1e-3) / 1e9
        d = plan.describe()
        out[key] = {
            "smem": TV_CONFIGS[key][0], "thr_load": d["load"]["thr"],
            "thr_store": d["store"]["thr"],
            "tuned": [d["load"]["tuned"], d["store"]["tuned"]],
            "vec_bytes": [d["load"]["vec_bytes"], d["store"]["vec_bytes"]],
            "smem_wavefronts_per_tile": [
                [d["load"]["smem_wavefronts"], d["load"]["smem_wavefronts_ideal"]],
                [d["store"]["smem_wavefronts"], d["store"]["smem_wavefronts_ideal"]]],
            "median_us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4),
            "isolated_us": round(iso[key] * 1e3, 2),
            "isolated_frac_of_peak": round(igbs / peak, 4)}
    return out


def measure_exchange(suite, args, torch, peak, world=4) -> dict:
    """The sharded relayout's device work on one GPU: the 4096x4096 fp32
    transpose with rows sharded over `world` ranks on both sides.  Every
    rank's pack (one copy for all peers) and unpack run on this device, each
    rank on its own stream as the ranks of a real run are separate GPUs
    (every pack joined before any box moves), with device-to-device copies
    of the boxes standing in for the all-to-all (a collective on several
    GPUs); reported as the bytes all of them read and write over the time
    of all of them.  The packs and unpacks are also timed one after another
    on one stream (`pack_unpack_serial_us_per_pass`)."""
    it = next((i for i in suite.items if i["name"] == "C2"), None)
    if it is None:
        return {}
    lm = suite.lm
    eb = it["w"].elem_bytes
    src = lm.Layout.parse("(4096,4096):(4096,1)")
    dst = lm.Layout.parse("(4096,4096):(1,4096)")
    xs = [lm.Exchange(src, dst, eb, r, world) for r in range(world)]
    sizes = [x.sizes() for x in xs]
    total = 4096 * 4096 * eb
    buf_in = it["src"][:total]
    buf_out = it["dst"][:total]
    send = torch.empty(total, dtype=torch.uint8, device=buf_in.device)
    soff = []       # byte offset of box (p, q) in the packed buffer
    off = 0
    for p in range(world):
        row = []
        for q in range(world):
            row.append(off)
            off += sizes[p]["send"][q] * eb
        soff.append(row)
    dsc = [x.describe() for x in xs]

    # rank p's packed buffer holds its boxes for peers 0..world-1; the
    # exchange hands rank q the q-th box of every sender, which here are
    # equal in size, so a receive buffer is a strided gather of the send
    # buffers -- replaced by unpacking each rank's boxes from where they
    # lie (the same bytes an all-to-all would deliver)
    recv = torch.empty(total, dtype=torch.uint8, device=buf_in.device)
    box = sizes[0]["send"][0] * eb
    one_copy = all(d["one_copy_per_side"] for d in dsc)

    ranks = [torch.cuda.Stream(device=buf_in.device) for _ in range(world)]

    def fork(concurrent):
        if concurrent:
            ev = torch.cuda.Event()
            ev.record()
            for st in ranks:
                st.wait_event(ev)

    def join(concurrent):
        if concurrent:
            cur = torch.cuda.current_stream()
            for st in ranks:
                ev = torch.cuda.Event()
                ev.record(st)
                cur.wait_event(ev)

    def on(k, concurrent):
        return (torch.cuda.stream(ranks[k]) if concurrent
                else contextlib.nullcontext())

    def one(exchange=True, concurrent=True):
        fork(concurrent)
        for p, x in enumerate(xs):
            o, n = dsc[p]["src_origin"] * eb, dsc[p]["src_local"] * eb
            with on(p, concurrent):
                lm.exchange_pack_all(x, buf_in[o:o + n],
                                     send[soff[p][0]:soff[p][0] + world * box])
        join(concurrent)   # every box packed before any moves
        fork(concurrent)
        for q, x in enumerate(xs):
            o, n = dsc[q]["dst_origin"] * eb, dsc[q]["dst_local"] * eb
            r = recv[q * world * box:(q + 1) * world * box]
            with on(q, concurrent):
                if exchange:
                    for p in range(world):  # the exchange, as device copies
                        r[p * box:(p + 1) * box].copy_(
                            send[soff[p][q]:soff[p][q] + box])
                lm.exchange_unpack_all(x, r, buf_out[o:o + n])
        join(concurrent)

    def timed_pass(fn):
        """ms per pass of fn, replayed as one CUDA graph (the small
        launches of a pass would otherwise be timed at the host's launch
        rate)."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        run, how = fn, "eager launches"
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                fn()
            torch.cuda.synchronize()
            run, how = graph.replay, "one CUDA graph per pass"
        except Exception as exc:  # capture unsupported: time eager launches
            how = f"eager launches (graph capture failed: {type(exc).__name__})"
            torch.cuda.synchronize()
        passes = min(args.steps, 200)
        for _ in range(3):
            run()
        e0, e1 = (torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True))
        torch.cuda.synchronize()
        e0.record()
        for _ in range(passes):
            run()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / passes, how

    ms, how = timed_pass(one)
    # the library's part alone: every rank's pack and unpack
    ms_lib, _ = timed_pass(lambda: one(exchange=False))
    ms_serial, _ = timed_pass(lambda: one(exchange=False, concurrent=False))
    if lm.device_status() != 0:
        raise RuntimeError("a copy kernel gave up a bounded wait "
                           "(LM_E_TIMEOUT): the exchange run is invalid")
    # pack, stand-in exchange and unpack each read and write every element
    gbs = 3 * 2 * total / (ms * 1e-3) / 1e9
    gbs_lib = 2 * 2 * total / (ms_lib * 1e-3) / 1e9
    return {"workload": f"4096x4096 fp32 transpose, rows sharded over {world} "
                        "ranks on both sides, all ranks' packs and unpacks on "
                        "this GPU; the all-to-all stands in as device copies "
                        "of the boxes, timed too",
            "layout_copies_per_pass": 2 * world, "one_copy_per_side": one_copy,
            "launch": how,
            "us_per_pass": round(ms * 1e3, 2), "gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4),
            "pack_unpack_us_per_pass": round(ms_lib * 1e3, 2),
            "pack_unpack_gbs": round(gbs_lib, 1),
            "pack_unpack_frac_of_peak": round(gbs_lib / peak, 4),
            "ranks": "each rank on its own stream",
            "pack_unpack_serial_us_per_pass": round(ms_serial * 1e3, 2),
            "pack_unpack_serial_frac_of_peak": round(
                2 * 2 * total / (ms_serial * 1e-3) / 1e9 / peak, 4)}


# --------------------------------------------------------------------------
# host topology: which NUMA node the GPU hangs off, where pinned memory goes
# --------------------------------------------------------------------------

def _cpulist(text: str) -> list[int]:
    cpus = []
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.extend(range(int(a), int(b) + 1))
        else:
            cpus.append(int(part))
    return cpus


def _ranges(cpus) -> str:
    cpus = sorted(set(cpus))
    out, k = [], 0
    while k < len(cpus):
        j = k
        while j + 1 < len(cpus) and cpus[j + 1] == cpus[j] + 1:
            j += 1
        out.append(str(cpus[k]) if j == k else f"{cpus[k]}-{cpus[j]}")
        k = j + 1
    return ",".join(out)


def _read(path: str) -> str | None:
    try:
        with open(path) as fh:
            return fh.read().strip()
    except OSError:
        return None


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True,
                             timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    info = _read("/proc/cpuinfo") or ""
    fields = {}
    for ln in info.splitlines():
        if ":" in ln:
            k, v = ln.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    return (f"CPU implementer {fields.get('CPU implementer', '?')} part "
            f"{fields.get('CPU part', '?')}")


def host_topology(local: int) -> dict:
    """The GPU's PCI address and NUMA node, that node's CPUs, and this
    process's CPU affinity."""
    import torch
    props = torch.cuda.get_device_properties(local)
    bdf = None
    bus = getattr(props, "pci_bus_id", None)
    if bus is not None:
        bdf = (f"{getattr(props, 'pci_domain_id', 0) or 0:04x}:{bus:02x}:"
               f"{getattr(props, 'pci_device_id', 0) or 0:02x}.0")
    else:
        try:
            out = subprocess.run(
                ["nvidia-smi", f"--id={gpu_smi_id(local)}",
                 "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                capture_output=True, text=True, timeout=20).stdout.strip()
            dom, rest = out.lower().split(":", 1)
            bdf = f"{int(dom, 16):04x}:{rest}"
        except Exception:
            bdf = None
    node = -1
    if bdf:
        txt = _read(f"/sys/bus/pci/devices/{bdf}/numa_node")
        node = int(txt) if txt not in (None, "") else -1
    node_cpus = []
    if node >= 0:
        node_cpus = _cpulist(_read(
            f"/sys/devices/system/node/node{node}/cpulist") or "")
    aff = sorted(os.sched_getaffinity(0))
    return {"gpu_pci": bdf, "gpu_numa_node": node,
            "gpu_node_cpus": _ranges(node_cpus),
            "process_affinity": _ranges(aff), "nproc": len(aff),
            "cpu_model": cpu_model()}


def _set_mempolicy(node: int | None) -> bool:
    """Prefer `node` for this thread's page allocations (None: back to the
    default policy), by the set_mempolicy system call."""
    import ctypes
    import platform
    nr = {"x86_64": 238, "aarch64": 237}.get(platform.machine())
    if nr is None:
        return False
    libc = ctypes.CDLL(None, use_errno=True)
    if node is None:
        rc = libc.syscall(ctypes.c_long(nr), ctypes.c_int(0), None,
                          ctypes.c_ulong(0))
    else:
        mask = (ctypes.c_ulong * 2)()
        mask[node // 64] = 1 << (node % 64)
        rc = libc.syscall(ctypes.c_long(nr), ctypes.c_int(1), mask,
                          ctypes.c_ulong(129))      # MPOL_PREFERRED
    return rc == 0


def pinned_near_gpu(topo: dict, local: int, items) -> tuple[list, str]:
    """Pinned host tensors of the given sizes (and contents: an array or
    None), allocated and first written by a thread bound to the CPUs of the
    GPU's NUMA node with that node preferred for its pages."""
    import threading
    import torch
    res = {}

    def work():
        try:
            how = []
            node = topo["gpu_numa_node"]
            if node >= 0:
                # placement is best effort: a refused binding is noted and
                # the buffers are allocated all the same
                want = set(_cpulist(topo["gpu_node_cpus"]))
                cpus = want & set(os.sched_getaffinity(0))
                try:
                    if cpus:
                        os.sched_setaffinity(0, cpus)
                        how.append(f"allocated by a thread bound to CPUs "
                                   f"{_ranges(cpus)} of node {node}")
                    else:
                        how.append(f"no CPU of node {node} in this "
                                   "process's affinity")
                except OSError as exc:
                    how.append(f"CPU binding refused ({exc.strerror})")
                try:
                    if _set_mempolicy(node):
                        how.append(f"pages preferred on node {node}")
                    else:
                        how.append("memory policy not set")
                except OSError:
                    how.append("memory policy not set")
            else:
                how.append("GPU NUMA node unknown: default placement")
            torch.cuda.set_device(local)
            out = []
            for n, content in items:
                t = torch.empty(n, dtype=torch.uint8, pin_memory=True)
                if content is not None:
                    t.numpy()[:] = content
                out.append(t)
            if node >= 0:
                _set_mempolicy(None)
            res["t"], res["how"] = out, "; ".join(how)
        except Exception as exc:       # reported by the caller
            res["err"] = exc

    th = threading.Thread(target=work)
    th.start()
    th.join()
    if "err" in res:
        raise res["err"]
    return res["t"], res["how"]


def measure_e2e(suite, args, torch, shards=4, topo=None) -> dict:
    """The same metric through the public API with host buffers: every step
    runs layout_copy_host -- upload of the source from pinned host memory,
    the copy, download of the destination into pinned host memory -- for
    every workload, each on its own stream so uploads and downloads share
    the two directions of the host link.  A workload whose shards
    (Plan(..., rank, world)) own disjoint source and destination ranges runs
    as `shards` shards, each moving only its ranges, so its transfers spread
    over several copy engines.

    In the same run, the same uploads and downloads without the copies give
    the link's ceilings for these byte counts: uploads alone, downloads
    alone, and both at once (the end-to-end figure's own bound).  The host
    link is shared with the machine's other GPUs, so the four measurements
    alternate over E2E_ROUNDS rounds and each figure is its median round:
    a burst of outside traffic then weighs on the copies and their ceilings
    alike.  Pinned buffers are allocated near the GPU (pinned_near_gpu)."""
    steps = max(20, min(args.steps, 40))
    lm = suite.lm
    local = suite.items[0]["src"].device.index or 0
    topo = topo or host_topology(local)
    pinned, how = pinned_near_gpu(
        topo, local, [x for it in suite.items
                      for x in ((it["host"].size, it["host"]),
                                (it["dst"].numel(), None))])
    jobs, h2d, d2h, sharded, moves = [], 0, 0, [], []
    for k, it in enumerate(suite.items):
        hs, hd = pinned[2 * k], pinned[2 * k + 1]
        eb = it["w"].elem_bytes
        plans = [lm.Plan(it["S"], it["D"], eb, rank=r, world=shards)
                 for r in range(shards)]
        descs = [p.describe() for p in plans]
        src_moved = sum(d["src_range"][1] - d["src_range"][0] for d in descs)
        if not all(d["dst_own"] for d in descs) or src_moved > it["S"].cosize:
            plans, descs = [it["plan"]], [it["plan"].describe()]
        else:
            sharded.append(it["name"])
        whole = len(plans) == 1
        for p, d in zip(plans, descs):
            jobs.append((p, hs, hd, it["src"], it["dst"]))
            up = ((0, hs.numel()) if whole else
                  (d["src_range"][0] * eb, d["src_range"][1] * eb))
            down = (d["dst_range"][0] * eb, d["dst_range"][1] * eb)
            moves.append((hs, hd, it["src"], it["dst"], up, down))
            h2d += up[1] - up[0]
            d2h += down[1] - down[0]
    main = torch.cuda.current_stream()
    streams = [torch.cuda.Stream() for _ in jobs]

    def copies():
        for (p, hs, hd, sdev, ddev), st in zip(jobs, streams):
            lm.layout_copy_host(p, hs, hd, sdev, ddev, st)

    def transfers(up: bool, down: bool):
        def run():
            for (hs, hd, sdev, ddev, (u0, u1), (d0, d1)), st in zip(moves,
                                                                   streams):
                with torch.cuda.stream(st):
                    if up:
                        sdev[u0:u1].copy_(hs[u0:u1], non_blocking=True)
                    if down:
                        hd[d0:d1].copy_(ddev[d0:d1], non_blocking=True)
        return run

    def timed(fn) -> float:
        """ms per step of fn over `steps` steps, streams forked from and
        joined to the current stream around them."""
        def fork():
            ev = torch.cuda.Event()
            ev.record(main)
            for st in streams:
                st.wait_event(ev)

        def join():
            for st in streams:
                ev = torch.cuda.Event()
                ev.record(st)
                main.wait_event(ev)

        fork()
        fn()
        join()
        torch.cuda.synchronize()
        start, end = (torch.cuda.Event(enable_timing=True),
                      torch.cuda.Event(enable_timing=True))
        start.record(main)
        fork()
        for _ in range(steps):
            fn()
        join()
        end.record(main)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / steps

    rounds = {"copies": [], "up": [], "down": [], "both": []}
    for _ in range(E2E_ROUNDS):
        rounds["copies"].append(timed(copies))
        if lm.device_status() != 0:
            raise RuntimeError("a copy kernel gave up a bounded wait "
                               "(LM_E_TIMEOUT): the end-to-end run is "
                               "invalid")
        rounds["up"].append(timed(transfers(True, False)))
        rounds["down"].append(timed(transfers(False, True)))
        rounds["both"].append(timed(transfers(True, True)))

    def median(xs):
        return sorted(xs)[len(xs) // 2]

    ms, up_ms, down_ms, both_ms = (median(rounds[k]) for k in
                                   ("copies", "up", "down", "both"))
    gb = 1e9
    return {"ms": ms * steps, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "rounds": E2E_ROUNDS,
            "value_per_round": [round(suite.bytes_per_step / (m * 1e-3) / gb,
                                      1) for m in rounds["copies"]],
            "duplex_per_round": [round((h2d + d2h) / (m * 1e-3) / gb, 1)
                                 for m in rounds["both"]],
            "path": f"layout_copy_host, {len(jobs)} plans on their own "
                    f"streams ({', '.join(sharded) or 'none'} as {shards} "
                    "shards each)",
            "h2d_ceiling_gbs": round(h2d / (up_ms * 1e-3) / gb, 1),
            "d2h_ceiling_gbs": round(d2h / (down_ms * 1e-3) / gb, 1),
            "duplex_ceiling_gbs": round((h2d + d2h) / (both_ms * 1e-3) / gb,
                                        1),
            "transfers_only_value": round(
                suite.bytes_per_step / (both_ms * 1e-3) / gb, 1),
            "ceilings": "the same uploads and downloads on the same streams "
                        "without the copies, this run, alternating with the "
                        "copies' rounds: uploads alone, downloads alone, "
                        "both at once; transfers_only_value is the metric "
                        "for the last (the bound of value); each figure is "
                        "the median of its rounds",
            "pinned": how, "topology": topo}


# --------------------------------------------------------------------------
# the CPU oracle (baseline leg and reference arm)
# --------------------------------------------------------------------------

class OracleWindows:
    """The CPU oracle's copy over windows of each workload's logical
    indices (the same fraction of every workload, so a sample mirrors the
    suite's mix).  Buffers are full-size host arrays.  With threads > 1 each
    window is split into that many contiguous index ranges, copied by one
    thread each (numpy releases the interpreter lock inside the oracle's
    array operations, so the threads run on separate cores)."""

    def __init__(self, names, bufs):
        from oracle import layout_oracle as lo
        self.lo = lo
        self.names = names
        self.bufs = bufs
        self.exprs = {n: (lo.build(WORKLOADS[n].src), lo.build(WORKLOADS[n].dst))
                      for n in names}
        for _, out in bufs.values():   # map every page before timing
            out.fill(0)

    def run(self, frac: float, shift: int = 0, threads: int = 1):
        from concurrent.futures import ThreadPoolExecutor
        nbytes, elems = 0.0, 0
        pool = ThreadPoolExecutor(threads) if threads > 1 else None
        t0 = time.perf_counter()
        for name in self.names:
            S, D = self.exprs[name]
            eb = WORKLOADS[name].elem_bytes
            inp, out = self.bufs[name]
            n = max(1, min(S.size, int(S.size * frac)))
            start = (shift * n) % max(1, S.size - n + 1)

            def part(k, S=S, D=D, eb=eb, inp=inp, out=out, n=n, start=start):
                a = start + n * k // threads
                b = start + n * (k + 1) // threads
                if b > a:
                    idx = np.arange(a, b, dtype=np.int64)
                    self.lo.copy(S, D, inp, out, eb, indices=idx)

            if pool is None:
                part(0)
            else:
                list(pool.map(part, range(threads)))
            nbytes += ALGO_BYTES[name] * n / S.size
            elems += n
        dt = time.perf_counter() - t0
        if pool is not None:
            pool.shutdown()
        return dt, nbytes, elems

    def calibrate(self, seconds: float, least: float = 2.0 ** -20,
                  threads: int = 1) -> float:
        """Fraction of every workload that takes about `seconds` (at least
        `least`): two probe windows give the fixed cost and the cost per
        fraction."""
        p1, p2 = 2.0 ** -11, 2.0 ** -7
        t1, _, _ = self.run(p1, threads=threads)
        t2, _, _ = self.run(p2, threads=threads)
        per = max((t2 - t1) / (p2 - p1), 1e-6)
        fixed = max(t1 - per * p1, 0.0)
        f = min(1.0, max(least, (seconds - fixed) / per))
        # large windows cost more per element than the probes (fresh
        # temporaries): one run at the estimate corrects it
        t, _, _ = self.run(f, threads=threads)
        return min(1.0, max(least, f * seconds / max(t, 1e-4)))


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_baseline(suite) -> dict:
    """The oracle as it stands, on this host: one core, then every core of
    the process's affinity (the same loop over contiguous index ranges, one
    thread each), each on a window of about 8 s of work."""
    bufs = {it["name"]: (it["host"],
                         np.zeros(it["dst"].numel(), dtype=np.uint8))
            for it in suite.items}
    ow = OracleWindows(BENCH_SUITE, bufs)
    legs = {}
    ncores = host_cores()
    for key, threads in (("cores_1", 1), ("cores_all", ncores)):
        frac = ow.calibrate(8.0, least=2.0 ** -7, threads=threads)
        secs, nbytes, elems = ow.run(frac, threads=threads)
        legs[key] = {
            "value": round(nbytes / secs / 1e9, 3), "threads": threads,
            "sample": f"numpy oracle copy of {frac:.4f} of every workload's "
                      f"logical indices (one contiguous window each, split "
                      f"into {threads} ranges), {elems} elements in "
                      f"{secs:.1f} s"}
    return {"value": legs["cores_all"]["value"], "unit": UNIT,
            "cores": ncores, "kind": "oracle",
            "sample": legs["cores_all"]["sample"],
            "cores_1": legs["cores_1"], "cores_all": legs["cores_all"],
            "nproc": ncores, "cpu_model": cpu_model()}


def run_reference(args) -> dict | None:
    """The reference arm: the CPU oracle as it stands, on every host core of
    this process (contiguous index ranges, one thread each), each step a
    window of every workload sized so the whole run takes about a minute."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    from oracle import layout_oracle as lo
    bufs = {}
    for name in BENCH_SUITE:
        w = WORKLOADS[name]
        S, D = lo.build(w.src), lo.build(w.dst)
        bufs[name] = (seeded_bytes(w.values, w.dtype, lo.cosize(S), w.seed),
                      np.zeros(lo.cosize(D) * w.elem_bytes, dtype=np.uint8))
    ow = OracleWindows(BENCH_SUITE, bufs)
    threads = host_cores()
    per_step = 60.0 / (args.steps + args.warmup)
    frac = ow.calibrate(per_step, threads=threads)
    for k in range(args.warmup):
        ow.run(frac, shift=k, threads=threads)
    secs, nbytes, elems = 0.0, 0.0, 0
    for k in range(args.steps):
        t, b, e = ow.run(frac, shift=args.warmup + k, threads=threads)
        secs += t
        nbytes += b
        elems += e
    gbs = nbytes / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4),
        "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / max(args.steps, 1), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": "synthetic",
        "config": {"workload": "relayout suite C2+C3+C4+C5a+C5b, one "
                               "layout_copy each per step",
                   "sample_fraction_per_step": frac},
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT,
                         "cores": threads, "kind": "oracle",
                         "sample": f"{frac:.2e} of every workload per step, "
                                   f"{elems} logical indices in {secs:.1f} s, "
                                   f"{threads} threads over contiguous index "
                                   "ranges",
                         "nproc": threads, "cpu_model": cpu_model()},
        "e2e": {"value": round(gbs, 4), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workloads", default="",
                    help="comma-separated subset of the suite (profiling)")
    ap.add_argument("--e2e-shards", type=int, default=4,
                    help="shards per workload in the end-to-end figure")
    ap.add_argument("--quick", action="store_true",
                    help="skip the clock sampler, e2e and CPU legs (profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_native(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

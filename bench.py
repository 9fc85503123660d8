"""Benchmark: the convolution hot path on GB300, one JSON line on stdout.

One step = 16 passes of the whole hot path over 16 batches: each of the five
workloads (conv1d fp32 NCL, 1x1 NHWC bf16, dense 3x3 NHWC bf16, depthwise 3x3
stride-2 NHWC bf16, 3x3 stride-2 dgrad NHWC bf16) is run through the C ABI on
each of 16 copies of its operands, resident in HBM, as one group of 16
back-to-back launches per workload.  The copies of each workload but the tiny
conv1d one together exceed 2.5x L2, so every launch reads inputs that have been
evicted since their last use (inputs larger than L2; no flush kernel runs
between launches).  CUDA events sit between the groups on the launching
stream; a kernel's time is its group's time over 16.  ``value`` is the step's
aggregate TFLOP/s (algorithmic flops of all launches / step time);
per-workload TFLOP/s, GB/s and roofline fractions are in ``per_config``;
``roofline`` describes the kernel with the largest share of the step.

``--impl reference`` times the FP64 CPU oracle instead (the reference arm: a
bounded sample of every workload per step, on the host cores).

Multi-GPU (torchrun): each rank runs the same step on its own GPU (replicas,
weak scaling, no collective on the data path); the step time is the max over
ranks and ``value`` the work of all ranks over that time.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
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

from synth.workloads import EXTRA_WORKLOADS, WORKLOADS, make_inputs  # noqa: E402

METRIC = "conv fwd/dgrad TFLOP/s (or GB/s) per config and % of roofline on 1 GB300"
UNIT = "TFLOP/s"
COPIES = 16  # operand copies per workload = passes over the hot path per step
WORKLOAD_NAME = "conv hot path: 5 workloads x 16 batches per step (conv1d f32, 1x1, dense 3x3, depthwise 3x3 s2, dgrad 3x3 s2)"


def max_over_ranks(value: float, device=None) -> float:
    """The largest of every rank's value (a job's time is its slowest rank's); the value itself when
    no process group is running or it has one rank."""
    import torch
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job TFLOP/s: every rank's algorithmic flops over the slowest rank's time (weak scaling)."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "sm_max_mhz") if k in m})
        p["source"] = "measured"
    return p


def out_hw(wl):
    """Output extent of a workload (the forward's), from the output-size rule."""
    res = []
    for i in range(wl.spatial_dims):
        eff = (wl.k[i] - 1) * wl.dil[i] + 1
        res.append((wl.in_size[i] + 2 * wl.pad[i] - eff) // wl.stride[i] + 1)
    return res


def work(wl):
    """(algorithmic flops, compulsory bytes) of one launch of a workload."""
    o = int(np.prod(out_hw(wl)))
    taps = int(np.prod(wl.k))
    flops = 2 * wl.n * o * wl.c_out * (wl.c_in // wl.groups) * taps
    es = 4 if wl.dtype == "f32" else 2
    x = wl.n * int(np.prod(wl.in_size)) * wl.c_in * es
    y = wl.n * o * wl.c_out * es
    w = wl.c_out * (wl.c_in // wl.groups) * taps * es
    b = 4 * wl.c_out if wl.bias else 0
    return flops, x + y + w + b


def desc_for(gb, wl):
    one = (lambda t: t[0]) if wl.spatial_dims == 1 else (lambda t: tuple(t))
    return gb.make_desc(wl.n, wl.c_in, wl.c_out, one(wl.in_size), one(wl.k), one(wl.stride), one(wl.pad),
                        one(wl.dil), wl.groups, spatial_dims=wl.spatial_dims, layout=wl.layout,
                        wlayout=wl.wlayout, dtype=wl.dtype)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                mhz.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def source_digest(kernel_file: str) -> str:
    src = os.path.join(ROOT, "convolution_conv_fwd_gb300", "csrc", kernel_file)
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def traffic_record(kernel_file: str, workload: str):
    """(DRAM bytes per launch, note) of a workload's kernel from profiles/traffic.json, which only
    ``--record-traffic`` writes (from an ncu capture).  The bytes are None, with the reason in the
    note, when there is no record or the kernel source changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_JSON):
        return None, "no ncu traffic record"
    rec = json.load(open(TRAFFIC_JSON)).get(workload)
    if rec is None or rec.get("kernel_file") != kernel_file:
        return None, "no ncu traffic record for this workload"
    if rec.get("source_sha16") != source_digest(kernel_file):
        return None, "kernel source changed since the ncu capture (%s)" % rec.get("source_sha16")
    return float(rec["dram_bytes_per_launch"]), "ncu capture at source %s" % rec["source_sha16"]


_NCU_UNITS = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12}


def ncu_dram_bytes(csv_path: str, kernel_regex: str):
    """Mean dram__bytes_read.sum + dram__bytes_write.sum per captured launch of kernels matching
    kernel_regex, from an ``ncu --metrics ... --csv --log-file`` file."""
    import csv
    import re
    per = {}
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        name = row.get("Metric Name", "")
        if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        if not re.search(kernel_regex, row.get("Kernel Name", "")):
            continue
        scale = _NCU_UNITS.get(row.get("Metric Unit", "byte").strip().lower())
        if scale is None:
            raise ValueError("unknown ncu unit %r" % row.get("Metric Unit"))
        val = float(row["Metric Value"].replace(",", "")) * scale
        per[row["ID"]] = per.get(row["ID"], 0.0) + val
    if not per:
        raise ValueError("no DRAM byte counters for kernels matching %r in %s" % (kernel_regex, csv_path))
    return sum(per.values()) / len(per), len(per)


def record_traffic(csv_path: str, workload: str, kernel_regex: str, command: str):
    """Write one workload's DRAM traffic per launch into profiles/traffic.json (machine-written;
    keyed by the workload and the hash of its kernel's source at the time of the capture)."""
    from synth.workloads import BY_NAME
    import convolution_conv_fwd_gb300 as gb
    wl = BY_NAME[workload]
    op = {"fwd": gb.GBCONV_OP_FWD, "dgrad": gb.GBCONV_OP_BWD_DATA, "wgrad": gb.GBCONV_OP_BWD_FILTER}[wl.op]
    kfile = KERNEL_FILE[gb.gbconv_select(desc_for(gb, wl), op)]
    nbytes, launches = ncu_dram_bytes(csv_path, kernel_regex)
    data = json.load(open(TRAFFIC_JSON)) if os.path.exists(TRAFFIC_JSON) else {}
    data[workload] = {"kernel_file": kfile, "source_sha16": source_digest(kfile), "kernel_regex": kernel_regex,
                      "dram_bytes_per_launch": round(nbytes), "launches_captured": launches,
                      "algorithmic_bytes": work(wl)[1], "command": command}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({workload: data[workload]}))


KERNEL_FILE = {"direct": "direct.cu", "depthwise": "depthwise.cu", "pointwise": "pointwise.cu",
               "implicit": "implicit.cu", "dgrad": "implicit.cu", "direct_dgrad": "direct.cu",
               "depthwise_dgrad": "depthwise.cu", "direct_wgrad": "wgrad.cu", "wgrad": "wgrad_tc.cu",
               "smallgroup": "smallgroup.cu", "smallgroup_dgrad": "smallgroup.cu"}

# Families whose arithmetic runs on the CUDA cores (fp32 FMA), not the tensor cores.
CUDA_CORE_FAMILIES = {"direct", "direct_dgrad", "direct_wgrad", "depthwise", "depthwise_dgrad", "smallgroup",
                      "smallgroup_dgrad"}


def fp32_peak_tflops(sms: int, sm_mhz: float) -> float:
    """FP32 FMA peak from unit counts: 128 fp32 lanes per SM, one FMA (2 flops) per lane per clock."""
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def run_gpu(args, rank, world, local_rank):
    import torch
    import convolution_conv_fwd_gb300 as gb

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    pk = peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    pk["fp32_tflops"] = fp32_peak_tflops(props.multi_processor_count, pk.get("sm_max_mhz", 2070.0))

    def make_case(wl):
        inp = make_inputs(wl)
        d = desc_for(gb, wl)
        xs, ws, ys = gb.desc_shapes(d)
        if wl.dtype == "bf16":
            def t(bits):
                return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
            # operands: (x, w) forward, (dy, w) input gradient, (x, dy) weight gradient
            src = t(inp["g_bits"] if wl.op == "dgrad" else inp["x_bits"])
            w = t(inp["g_bits"] if wl.op == "wgrad" else inp["w_bits"])
            dt = torch.bfloat16
        else:
            src = torch.from_numpy(inp["g"] if wl.op == "dgrad" else inp["x"]).to(dev)
            w = torch.from_numpy(inp["g"] if wl.op == "wgrad" else inp["w"]).to(dev)
            dt = torch.float32
        b = torch.from_numpy(inp["b"]).to(dev) if "b" in inp else None
        out_shape = {"dgrad": xs, "wgrad": ws}.get(wl.op, ys)
        op = {"fwd": gb.GBCONV_OP_FWD, "dgrad": gb.GBCONV_OP_BWD_DATA, "wgrad": gb.GBCONV_OP_BWD_FILTER}[wl.op]
        family = gb.gbconv_select(d, op)
        flops, nbytes = work(wl)
        # COPIES copies of every operand: a launch's inputs were last touched a full rotation
        # earlier, with more than 2x L2 of other traffic in between (every workload but the tiny
        # conv1d one has COPIES x its footprint > 2.5x L2), so every launch reads them from HBM
        # with no flush kernel (and no flush write-back) between launches.
        per_copy = (src.numel() * src.element_size() + w.numel() * w.element_size()
                    + int(np.prod(out_shape)) * src.element_size() + (0 if b is None else b.numel() * 4))
        reps = COPIES
        copies = [(src.clone(), w.clone(), None if b is None else b.clone(), torch.empty(out_shape, dtype=dt, device=dev))
                  for _ in range(reps)]
        # the weight gradient's scratch: one buffer serves every copy (launches are stream-ordered)
        wsp = (torch.empty((gb.gbconv_bwd_filter_workspace(d),), dtype=torch.uint8, device=dev)
               if wl.op == "wgrad" else None)
        return dict(wl=wl, d=d, copies=copies, family=family, flops=flops, bytes=nbytes, host=inp,
                    l2_resident=reps * per_copy < int(2.5 * l2), workspace=wsp)

    cases = [make_case(wl) for wl in WORKLOADS]

    def launch(c, k):
        s = stream.cuda_stream
        src, w, b, out = c["copies"][k]
        if c["wl"].op == "dgrad":
            rc = gb.gbconv_bwd_data(c["d"], src.data_ptr(), w.data_ptr(), out.data_ptr(), s)
        elif c["wl"].op == "wgrad":
            wsp = c["workspace"]
            rc = gb.gbconv_bwd_filter(c["d"], src.data_ptr(), w.data_ptr(), out.data_ptr(), None, wsp.data_ptr(),
                                      wsp.numel(), s)
        else:
            rc = gb.gbconv_fwd(c["d"], src.data_ptr(), w.data_ptr(), None if b is None else b.data_ptr(),
                               out.data_ptr(), s)
        if rc != gb.GBCONV_OK:
            raise gb.GbconvError(rc, c["wl"].name)

    def step(events=None):
        # One group per workload: one launch per copy, back to back on one stream.  Events sit
        # only between groups, so a kernel's time is its group's time over its launch count.
        for i, c in enumerate(cases):
            if events is not None and i == 0:
                events[0].record(stream)
            for k in range(len(c["copies"])):
                launch(c, k)
            if events is not None:
                events[i + 1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    gb.device_status()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(cases) + 1)] for _ in range(args.steps)]
    launches0 = gb.gbconv_kernels_launched()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = time.perf_counter()
        # A spin kernel first, so every later launch is queued before the GPU reaches it: the events
        # then bracket device time only, with no gaps from host-side launch latency.
        torch.cuda._sleep(int(3e8))
        for k in range(args.steps):
            step(evs[k])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    launches = gb.gbconv_kernels_launched() - launches0
    gb.device_status()
    group_ms = [statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps))
                for i in range(len(cases))]
    per_kernel_ms = [g / len(c["copies"]) for g, c in zip(group_ms, cases)]
    step_ms = max_over_ranks(statistics.mean(evs[k][0].elapsed_time(evs[k][-1]) for k in range(args.steps)), dev)

    def config_line(c, ms):
        # the slower of the flops at the dense bf16 tensor peak and the bytes at the copy bandwidth;
        # for a family that runs on the CUDA cores, also the flops at the fp32 FMA peak
        t_f = c["flops"] / (pk["bf16_tflops"] * 1e12)
        t_b = c["bytes"] / (pk["hbm_gbs"] * 1e9)
        t_a = c["flops"] / (pk["fp32_tflops"] * 1e12) if c["family"] in CUDA_CORE_FAMILIES else 0.0
        t_roof = max(t_f, t_b, t_a)
        bound = "alu" if t_a >= max(t_f, t_b) else ("tensor" if t_f >= t_b else "hbm")
        line = {"workload": c["wl"].name, "kernel": c["family"], "us": round(ms * 1e3, 3),
                "tflops": round(c["flops"] / (ms * 1e-3) / 1e12, 2),
                "gbs": round(c["bytes"] / (ms * 1e-3) / 1e9, 1),
                "bound": bound, "t_roof_us": round(t_roof * 1e6, 3),
                "roofline_frac": round(t_roof / (ms * 1e-3), 4),
                "launches_per_step": len(c["copies"]),
                "inputs": "L2 resident (too small to exceed L2)" if c["l2_resident"] else "from HBM"}
        if bound == "alu":
            line["roofline_frac_tensor_hbm"] = round(max(t_f, t_b) / (ms * 1e-3), 4)
        return line

    # ---------------------------------------------------------------- widened rows, timed the same way
    # Not part of the step (the step is the five configs above): the same grouped, back-to-back
    # timing over 16 rotating copies, after the step's timed region.
    extra = []
    for wl in EXTRA_WORKLOADS:
        c = make_case(wl)
        for k in range(len(c["copies"])):
            launch(c, k)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        torch.cuda._sleep(int(1e8))
        ev[0].record(stream)
        for i in range(args.steps):
            for k in range(len(c["copies"])):
                launch(c, k)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)) / len(c["copies"])
        extra.append(config_line(c, ms))
        del c
    gb.device_status()

    # ---------------------------------------------------------------- end to end through the public API
    e2e_ms, h2d, d2h = None, 0, 0
    host_cases = []
    for c in cases:
        src, w, b, out = c["copies"][0]
        hs = src.cpu().pin_memory()
        hw = w.cpu().pin_memory()
        hb = None if b is None else b.cpu().pin_memory()
        host_cases.append((c, hs, hw, hb))
        h2d += hs.numel() * hs.element_size() + hw.numel() * hw.element_size() + (0 if hb is None else hb.numel() * 4)
        d2h += out.numel() * out.element_size()
    # The five calls are independent: enqueued back to back, then every result is waited on.  The
    # largest host-to-device transfer goes first (while it streams, the host enqueues the rest, so the
    # link never waits for the host), the others by result size (a long copy back overlaps the later
    # calls' copies in instead of ending the step).
    nbytes = lambda t: t.numel() * t.element_size()
    biggest_in = max(nbytes(hc[1]) for hc in host_cases)
    host_cases.sort(key=lambda hc: (nbytes(hc[1]) < biggest_in, -nbytes(hc[0]["copies"][0][3])))

    def e2e_step():
        calls = [gb.conv_bwd_data_async(c["d"], hs, hw) if c["wl"].op == "dgrad" else
                 gb.conv_fwd_async(c["d"], hs, hw, hb) for c, hs, hw, hb in host_cases]
        for h in calls:
            h.wait()
    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    # Host-timed: as timeit does, Python's cyclic garbage collector is run before the timed steps and
    # kept off during them (a full collection of this process's objects takes tens of ms).
    gc.collect()
    gc.disable()
    e2e_steps = []  # each step ends with every result waited on, so the host clock brackets it
    # At least 100 steps (about 0.17 s): the mean of a host-timed loop of 20 steps (33 ms) moved by
    # tens of percent with one pause of the host.
    e2e_n = max(args.steps, 100)
    try:
        t0 = time.perf_counter()
        for _ in range(e2e_n):
            ts = time.perf_counter()
            e2e_step()
            e2e_steps.append((time.perf_counter() - ts) * 1e3)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / e2e_n, dev)
    finally:
        gc.enable()

    total_flops = sum(c["flops"] for c in cases)
    step_flops = sum(c["flops"] * len(c["copies"]) for c in cases)

    per = [config_line(c, ms) for c, ms in zip(cases, per_kernel_ms)]
    dom = max(range(len(cases)), key=lambda i: group_ms[i])
    dc, dms = cases[dom], per_kernel_ms[dom]
    if per[dom]["bound"] == "hbm":
        achieved, peak, unit = dc["bytes"] / (dms * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s"
    elif per[dom]["bound"] == "alu":
        achieved, peak, unit = dc["flops"] / (dms * 1e-3) / 1e12, pk["fp32_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = dc["flops"] / (dms * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s"
    traffic, traffic_note = traffic_record(KERNEL_FILE[dc["family"]], dc["wl"].name)
    roof = {"bound": per[dom]["bound"], "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": traffic_note,
            "kernel": dc["family"], "workload": dc["wl"].name,
            "algorithmic_bytes": dc["bytes"], "algorithmic_flops": dc["flops"],
            "peak_source": (pk["source"] + " (burst)") if per[dom]["bound"] != "alu" else
                           "fp32 FMA from unit counts: SMs x 128 lanes x 2 flops x max SM clock"}
    value = job_rate(world, step_flops, step_ms)
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME,
                   "l2": "not flushed: inputs larger than L2 -- each workload rotates over operand copies totalling "
                         "> 2.5x L2, so every launch reads its inputs from HBM",
                   "launch": "back-to-back on one stream, programmatic dependent launch; events between workload groups",
                   "inputs": "seeded SplitMix64/Box-Muller, bf16 RNE; conv1d workload fp32",
                   # every launch of the step at its roofline time, over the measured step time
                   "step_roofline_frac": round(sum(p["t_roof_us"] * p["launches_per_step"] for p in per)
                                               / (step_ms * 1e3), 4),
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "per_config": per,
        "extra_configs": extra,
        "roofline": roof,
        "e2e": {"value": round(job_rate(world, total_flops, e2e_ms), 4), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "steps": e2e_n,
                "step_ms": {"min": round(min(e2e_steps), 3), "median": round(statistics.median(e2e_steps), 3),
                            "max": round(max(e2e_steps), 3)},
                "path": "one batch of each workload per step from pinned host tensors through the public host "
                        "calls (conv_fwd_async / conv_bwd_data_async: batch slices pipelined through a device "
                        "staging buffer), the five calls enqueued back to back and every result waited on inside "
                        "the timed region; largest transfer in first, then by result size"},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "wall_s_timed": round(wall, 3),
    }
    return res, cases


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_sample(target_s: float, cases_host, threads: int = 1):
    """Time the FP64 oracle on a bounded, strided sample of every workload's outputs, on `threads`
    host threads (disjoint slices of the sample; the oracle's C loops run without the GIL)."""
    import oracle
    from tests.helpers import oracle_conv  # the same shape mapping the tests use
    oracle.build()
    per_point = []
    for wl, inp in cases_host:
        c = oracle_conv(wl)
        if wl.op == "dgrad":
            n, ch, h, w = wl.n, wl.c_in, wl.in_size[0], wl.in_size[1]
            iters = (wl.c_out // wl.groups) * int(np.prod(wl.k))
        else:
            oh = out_hw(wl)
            n, ch = wl.n, wl.c_out
            h, w = (oh[0], oh[1]) if wl.spatial_dims == 2 else (1, oh[0])
            iters = (wl.c_in // wl.groups) * int(np.prod(wl.k))
        per_point.append((wl, inp, c, (n, ch, h, w), iters))
    # calibrate: a small sample of the heaviest workload
    budget_iters = None
    wl, inp, c, shp, iters = max(per_point, key=lambda p: p[4])
    probe = 2000 * threads
    t = _time_points(wl, inp, c, shp, probe, threads)
    rate = probe * iters / max(t, 1e-6)  # inner iterations per second
    budget_iters = rate * target_s
    total_flops, total_s, points = 0.0, 0.0, {}
    for wl, inp, c, shp, iters in per_point:
        outputs = int(np.prod(shp))
        count = int(min(outputs, max(256, budget_iters / len(per_point) / iters)))
        dt = _time_points(wl, inp, c, shp, count, threads)
        flops, _ = work(wl)
        total_flops += flops * count / outputs
        total_s += dt
        points[wl.name] = count
    return total_flops, total_s, points


def _time_points(wl, inp, c, shp, count, threads=1):
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    n, ch, h, w = shp
    total = n * ch * h * w
    stride = max(1, total // count)
    flat = (np.arange(count, dtype=np.int64) * stride) % total
    idx = np.stack(np.unravel_index(flat, (n, ch, h, w)), axis=1).astype(np.int64)

    def run(part):
        if wl.op == "dgrad":
            oracle.conv_dgrad_points(c, inp["g"], inp["w"], part)
        else:
            oracle.conv_fwd_points(c, inp["x"], inp["w"], inp.get("b"), part)

    if threads <= 1:
        t0 = time.perf_counter()
        run(idx)
        return time.perf_counter() - t0
    parts = np.array_split(idx, threads)
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        list(pool.map(run, parts))
        return time.perf_counter() - t0


def run_reference(args):
    """The reference arm: the FP64 oracle on the host cores, one bounded sample per step."""
    cases_host = [(wl, make_inputs(wl)) for wl in WORKLOADS]
    cores = host_cores()
    for _ in range(args.warmup):
        cpu_sample(0.5, cases_host, cores)
    flops, secs = 0.0, 0.0
    points = {}
    for _ in range(args.steps):
        f, s, points = cpu_sample(args.ref_seconds_per_step, cases_host, cores)
        flops += f
        secs += s
    value = flops / secs / 1e12
    sample = "strided sample of every workload's outputs per step, %s points" % json.dumps(points)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME}, "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def profile_workload(name: str, reps: int):
    """Run one workload `reps` times through the C ABI (no timing, no oracle): the target of ncu captures."""
    import torch
    import convolution_conv_fwd_gb300 as gb
    from synth.workloads import BY_NAME
    wl = BY_NAME[name]
    inp = make_inputs(wl)
    d = desc_for(gb, wl)

    def dev(key):
        if wl.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(inp[key + "_bits"]).view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(inp[key]).cuda()
    b = torch.from_numpy(inp["b"]).cuda() if "b" in inp else None
    if wl.op == "wgrad":
        x, g = dev("x"), dev("g")
        wsp = torch.empty((gb.gbconv_bwd_filter_workspace(d),), dtype=torch.uint8, device="cuda")
        for _ in range(reps):
            gb.conv_bwd_filter(d, x, g, workspace=wsp)
        gb.device_status()
        print("ran", name, reps, "times")
        return
    w = dev("w")
    src = dev("g" if wl.op == "dgrad" else "x")
    for _ in range(reps):
        if wl.op == "dgrad":
            gb.conv_bwd_data(d, src, w)
        else:
            gb.conv_fwd(d, src, w, b)
    gb.device_status()
    print("ran", name, reps, "times")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gbconv", choices=["gbconv", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle work for the cpu_baseline sample")
    ap.add_argument("--ref-seconds-per-step", type=float, default=3.0)
    ap.add_argument("--profile-workload", default=None,
                    help="run only this workload --steps times through the C ABI and exit (for ncu captures)")
    ap.add_argument("--record-traffic", nargs=4, metavar=("NCU_CSV", "WORKLOAD", "KERNEL_REGEX", "COMMAND"),
                    help="write the workload's DRAM bytes per launch from an ncu --metrics "
                         "dram__bytes_read.sum,dram__bytes_write.sum --csv log into profiles/traffic.json")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(*args.record_traffic)
        return
    if args.profile_workload:
        profile_workload(args.profile_workload, args.steps)
        return
    if args.warmup < 3 and args.impl == "gbconv":
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res, cases = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        host = [(c["wl"], c["host"]) for c in cases]
        cores = host_cores()
        f1, s1, p1 = cpu_sample(args.cpu_seconds / 2, host, 1)
        fn, sn, pn = cpu_sample(args.cpu_seconds / 2, host, cores)
        res["cpu_baseline"] = {"value": fn / sn / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": "strided sample of every workload's outputs split over %d threads, %s points, "
                                         "%.1f s" % (cores, json.dumps(pn), sn),
                               "single_core": {"value": f1 / s1 / 1e12, "cores": 1,
                                               "sample": "%s points, %.1f s" % (json.dumps(p1), s1)}}
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

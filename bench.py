#!/usr/bin/env python
"""Throughput of the selective-scan layer core (forward + backward) on GB300.

One step = one forward (m3scan_fwd) and one backward (m3scan_bwd) of the
layer core over one batch of the workload, through the C ABI.  Prints ONE
JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Timing: inputs resident in HBM; each step is two CUDA-graph replays (forward
graph, backward graph) bracketed by CUDA events on the launching stream;
L2 is flushed (256 MiB memset, read back) between steps, outside the events.  The
end-to-end number repeats the step through the Python binding with inputs
copied from pinned host memory and results copied back inside the timed
region.  Multi-GPU runs are independent replicas (weak scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mamba_selective_scan_gb300.inputs import WORKLOADS, make_workload_inputs  # noqa: E402

METRIC = "selective-scan fwd+bwd Gelem/s (B*T*d_inner) and % of GB300 HBM roofline"
UNIT = "Gelem/s"
# the largest configuration that fits one GPU (134 M elements per step)
DEFAULT_WORKLOAD = "longseq_b1_t65536_d2048"
EXTRA_WORKLOADS = ("trainer_b8_t128_d512", "m130m_b8_t2048_d1536", "m2p8b_b4_t4096_d5120")
HBM_TARGET_GBS = 8000.0  # the roofline bandwidth the metric is defined with
L2_BYTES = 126 << 20     # GB300 L2 (the 256 MiB flush buffer is twice that)
ROOFLINE_CHUNK = 128     # chunk length of the metric's minimum-bytes formula
NS = 16


def algorithmic_bytes(batch, T, D, es, chunk=ROOFLINE_CHUNK):
    """Minimum bytes the fused design moves (per call), with checkpoints every
    `chunk` steps: forward reads x, delta_raw, z, B, C and writes gated and the
    checkpoints; backward reads x, delta_raw, z, d_gated, B, C and the
    checkpoints and writes d_x, d_delta_raw, dz, dB, dC (f32)."""
    E = batch * T * D
    nc = -(-T // chunk)
    bc = batch * T * 2 * NS
    ck = batch * nc * NS * D * 4
    fwd = E * 4 * es + bc * es + ck
    bwd = E * 7 * es + bc * es + bc * 4 + ck
    return fwd, bwd


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# FP32 lane operations the backward must execute per element (16 state lanes):
# recompute 4 per lane (delta*A, delta*u*B, the state update, nothing for the
# exponential itself), reverse pass 10 per lane (y, dh, dC and dB partials,
# the B sum, delta*A, the carry, dh*exp*h_prev, dA and the A-weighted sum),
# 32 adds of the cross-channel dB/dC reduction, about 35 per element of
# conv/SiLU/softplus/gate arithmetic.  Exponentials run on the MUFU pipe and
# are not counted.
BWD_FP32_OPS_PER_ELEM = 16 * (4 + 10) + 32 + 35
FP32_LANES_PER_SM = 128  # FFMA lanes per SM per clock on GB300 (measured 118-121)
GB300_SMS = 152


def alu_peak_gops():
    """FP32 lane-op peak of the whole GPU at the maximum SM clock."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            mhz = float(json.load(f).get("sm_max_mhz", 2070.0))
    except Exception:
        mhz = 2070.0
    return GB300_SMS * FP32_LANES_PER_SM * mhz * 1e6 / 1e9


# The translation units whose kernels (and launch logic) the forward and
# backward calls run; the decode and conv-backward unit is not among them.
SCAN_SOURCES = ("m3_api.cu", "m3_bwd.cu", "m3_bwd2.cu", "m3_common.cuh", "m3_fwd.cu")


def code_only(text):
    """C++/CUDA source with its comments removed and whitespace collapsed, so
    that an edit to comments alone leaves the hash unchanged (string literals
    here hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash():
    """Hash of the code (comments aside) of the forward/backward kernel
    sources the ncu traffic figures were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mamba_selective_scan_gb300", "csrc")
    for name in SCAN_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_sha256_16") != source_hash():
        return None
    return d.get("traffic", {}).get(workload, {}).get(kernel)


def traffic_from_launch_list(csv_path, workload):
    """The ncu_traffic.json record from an ncu launch list (the CSV of
    ``ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,
    dram__bytes_write.sum --csv``): DRAM bytes per launch of every m3_ kernel
    (read + write, averaged over its launches) and their sums over the
    forward's and the backward's kernels, keyed to the current kernel code."""
    import csv
    with open(csv_path, newline="") as f:
        rows = list(csv.reader(f))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    hdr = rows[hi]
    ki, ii = hdr.index("Kernel Name"), hdr.index("ID")
    mi, vi, ui = hdr.index("Metric Name"), hdr.index("Metric Value"), hdr.index("Metric Unit")
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per_launch = {}
    for r in rows[hi + 1:]:
        if len(r) <= vi or not r[mi].startswith("dram__bytes_"):
            continue
        name = r[ki].split("(")[0].replace("void ", "").strip()
        if not name.startswith("m3_"):
            continue
        key = (name, r[ii])
        per_launch[key] = per_launch.get(key, 0.0) + float(r[vi].replace(",", "")) * scale[r[ui]]
    sums = {}
    for (name, _), v in per_launch.items():
        tot, n = sums.get(name, (0.0, 0))
        sums[name] = (tot + v, n + 1)
    per = {k: int(tot / n) for k, (tot, n) in sums.items()}
    return {"note": "DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per call, summed "
                    "over the call's kernels, from one ncu launch list; valid only for the kernel "
                    "code with this hash",
            "source_sha256_16": source_hash(),
            "traffic": {workload: {"bwd": sum(v for k, v in per.items() if "bwd" in k),
                                   "fwd": sum(v for k, v in per.items() if "fwd" in k)}},
            "per_kernel_bytes_per_launch": per}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"m3scan_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                                     hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[k].lower().startswith("active"):
                    reasons.add(name)
        powers = [r["power"] for r in rows if r["power"] is not None]
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(powers) if powers else None}


# ---------------------------------------------------------------------------
# replicas: combining ranks
# ---------------------------------------------------------------------------

def max_over_ranks(dist, x, device=None):
    """The largest of a per-rank float over all ranks (x itself without a
    process group): the job is as slow as its slowest replica."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gelem_s(world, elems_per_rank_step, steps, total_ms):
    """Whole-job throughput: the elements every rank processed over the
    slowest rank's time."""
    return world * elems_per_rank_step * steps / (total_ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class Layer:
    """Device buffers, plan and captured graphs for one layer-core instance."""

    def __init__(self, torch, binding, tensors, chunk=0, segments=0, threads_per_channel=0,
                 deterministic=False):
        self.t = tensors
        x = tensors["x"]
        self.act = binding.M3_BF16 if x.dtype == torch.bfloat16 else binding.M3_F32
        Bsz, T, D = x.shape
        self.shape = (Bsz, T, D)
        self.segments, self.tpc = segments, threads_per_channel
        self.dims = binding.make_dims(Bsz, T, D, chunk=chunk, segments=segments,
                                      threads_per_channel=threads_per_channel,
                                      deterministic=deterministic)
        self.deterministic = deterministic
        self.plan = binding.m3scan_plan(self.dims, self.act)
        dev = x.device
        f32 = dict(dtype=torch.float32, device=dev)
        self.o = {
            "gated": torch.empty_like(x),
            "ckpt": torch.empty((Bsz, self.plan.n_chunks, NS, D), **f32),
            "d_x": torch.empty_like(x), "d_delta_raw": torch.empty_like(x),
            "dz": torch.empty_like(x),
            "dB": torch.empty((Bsz, T, NS), **f32), "dC": torch.empty((Bsz, T, NS), **f32),
            "d_conv_w": torch.empty((D, 4), **f32), "d_conv_b": torch.empty((D,), **f32),
            "d_dt_bias": torch.empty((D,), **f32), "d_a_log": torch.empty((D, NS), **f32),
            "dD": torch.empty((D,), **f32),
        }
        # zeroed: the library's status block at its start must begin at zero
        self.ws = torch.zeros(max(int(self.plan.workspace_bytes), 256), dtype=torch.uint8,
                              device=dev)
        self.binding = binding

    def fwd(self, stream):
        t, o, b = self.t, self.o, self.binding
        st = b.raw_fwd(self.dims, self.act, t["x"].data_ptr(), t["delta_raw"].data_ptr(),
                       t["z"].data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(),
                       t["conv_w"].data_ptr(), t["conv_b"].data_ptr(), t["dt_bias"].data_ptr(),
                       t["a_log"].data_ptr(), t["D"].data_ptr(), o["gated"].data_ptr(), None,
                       o["ckpt"].data_ptr(), self.ws.data_ptr(), self.ws.numel(), stream)
        if st != 0:
            raise b.M3Error(st, "m3scan_fwd")

    def bwd(self, stream):
        t, o, b = self.t, self.o, self.binding
        st = b.raw_bwd(self.dims, self.act, t["x"].data_ptr(), t["delta_raw"].data_ptr(),
                       t["z"].data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(),
                       t["conv_w"].data_ptr(), t["conv_b"].data_ptr(), t["dt_bias"].data_ptr(),
                       t["a_log"].data_ptr(), t["D"].data_ptr(), o["ckpt"].data_ptr(),
                       t["d_gated"].data_ptr(), o["d_x"].data_ptr(), o["d_delta_raw"].data_ptr(),
                       o["dz"].data_ptr(), None, o["dB"].data_ptr(), o["dC"].data_ptr(),
                       o["d_conv_w"].data_ptr(), o["d_conv_b"].data_ptr(),
                       o["d_dt_bias"].data_ptr(), o["d_a_log"].data_ptr(), o["dD"].data_ptr(),
                       self.ws.data_ptr(), self.ws.numel(), stream)
        if st != 0:
            raise b.M3Error(st, "m3scan_bwd")


def host_inputs_to_device(torch, inp, device):
    import numpy as np
    from mamba_selective_scan_gb300.inputs import bf16_bits
    out = {}
    for k, v in inp.arrays.items():
        if k in ("x", "delta_raw", "z", "B", "C", "d_gated") and inp.act == "bf16":
            out[k] = torch.from_numpy(bf16_bits(v).view(np.int16)).view(torch.bfloat16).to(device)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(device)
    return out


def device_inputs(torch, w, device, seed_offset=0):
    """Inputs drawn on the device with the recipe's distributions (used for
    the large extra workloads, where drawing with NumPy on the host would
    dominate the run time)."""
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * (w.seed + 1) + seed_offset)
    Bsz, T, D = w.batch, w.seq_len, w.d_inner
    act = torch.bfloat16 if w.act == "bf16" else torch.float32
    f32 = dict(dtype=torch.float32, device=device)

    def normal(shape, std=1.0):
        return (torch.randn(shape, generator=g, **f32) * std).to(act)

    def softplus_inv(y):
        return torch.log(torch.expm1(y.double())).float()
    t = {"x": normal((Bsz, T, D)), "z": normal((Bsz, T, D)), "d_gated": normal((Bsz, T, D))}
    t["conv_w"] = torch.rand((D, 4), generator=g, **f32) - 0.5
    dt_bias = softplus_inv(0.001 + 0.099 * torch.rand((D,), generator=g, **f32))
    if w.slow_delta:
        tgt = 0.001 + 0.009 * torch.rand((Bsz, T, D), generator=g, **f32)
        t["delta_raw"] = (softplus_inv(tgt) - dt_bias).to(act)
        del tgt
    else:
        t["delta_raw"] = normal((Bsz, T, D), 0.5)
    t["dt_bias"] = dt_bias
    t["B"] = normal((Bsz, T, NS))
    t["C"] = normal((Bsz, T, NS))
    t["conv_b"] = torch.zeros((D,), **f32)
    t["a_log"] = torch.log(torch.arange(1, NS + 1, **f32)).repeat(D, 1).contiguous()
    t["D"] = torch.ones((D,), **f32)
    return t


def capture(torch, layer_list, stream):
    """Capture the forward of every layer (in order) and the backward (in
    reverse order) as two CUDA graphs."""
    gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gf, stream=stream):
        for L in layer_list:
            L.fwd(torch.cuda.current_stream().cuda_stream)
    with torch.cuda.graph(gb, stream=stream):
        for L in reversed(layer_list):
            L.bwd(torch.cuda.current_stream().cuda_stream)
    return gf, gb


def flush_l2(torch, flush):
    """Evict L2 before a timed step: write a buffer twice the L2's size, then
    read it back, so that the lines it leaves in L2 are clean and no
    write-back of the flush lands inside the timed region."""
    flush.zero_()
    torch.amax(flush)


def time_steps(torch, gf, gb, steps, flush):
    """Per-step forward and backward device times (ms) with L2 flushed
    before every step."""
    s = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush_l2(torch, flush)
        e0, e1, e2 = ev[i]
        e0.record(s)
        gf.replay()
        e1.record(s)
        gb.replay()
        e2.record(s)
    torch.cuda.synchronize()
    f = [a.elapsed_time(b) for a, b, _ in ev]
    bw = [b.elapsed_time(c) for _, b, c in ev]
    return f, bw


def gpu_arm(args):
    import torch
    from mamba_selective_scan_gb300 import binding, build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if rank == 0 or world == 1:
        build.build()
    if dist is not None:
        dist.barrier()
    binding.load()

    w = WORKLOADS[args.workload]
    es = 2 if w.act == "bf16" else 4
    inp = make_workload_inputs(args.workload)
    tensors = host_inputs_to_device(torch, inp, device)
    layer = Layer(torch, binding, tensors, chunk=args.chunk, segments=args.segments,
                  threads_per_channel=args.threads_per_channel, deterministic=args.deterministic)
    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    # warm-up (eager), then capture
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            layer.fwd(stream.cuda_stream)
            layer.bwd(stream.cuda_stream)
    torch.cuda.synchronize()
    gf, gb = capture(torch, [layer], stream)
    for _ in range(args.warmup):
        gf.replay()
        gb.replay()
    torch.cuda.synchronize()

    # keep the GPU busy briefly so the clock samples see steady state
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + 0.3
    while time.time() < t_end:
        for _ in range(20):
            gf.replay()
            gb.replay()
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    f_ms, b_ms = time_steps(torch, gf, gb, args.steps, flush)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()

    total_ms = max_over_ranks(dist, sum(f_ms) + sum(b_ms), device)
    E = w.elems
    value = job_gelem_s(world, E, args.steps, total_ms)
    fwd_avg = sum(f_ms) / len(f_ms)
    bwd_avg = sum(b_ms) / len(b_ms)
    fwd_med = statistics.median(f_ms)
    bwd_med = statistics.median(b_ms)
    step_med = statistics.median([a + b for a, b in zip(f_ms, b_ms)])
    fb, bb = algorithmic_bytes(w.batch, w.seq_len, w.d_inner, es)
    peak, peak_kind = measured_peaks()
    step_s = (fwd_avg + bwd_avg) * 1e-3
    # The roofline of the metric: the minimum bytes the fused method moves
    # (checkpoints every 128 steps) over the measured HBM copy bandwidth, for
    # the dominant call (the backward: aggregate, main and any finishing
    # kernels of one m3scan_bwd, timed by CUDA events around its graph).
    bwd_achieved = bb / (bwd_avg * 1e-3) / 1e9
    alu_peak = alu_peak_gops()
    bwd_gops = BWD_FP32_OPS_PER_ELEM * E / (bwd_avg * 1e-3) / 1e9
    parts = (["aggregate"] if int(layer.plan.bwd_segments) > 1 else []) + ["main"]
    parts += ["tail", "dB/dC sum"][:max(0, int(layer.plan.bwd_launches) - len(parts))]
    bwd_kernels = " + ".join(parts) + (" kernels" if len(parts) > 1 else " kernel")
    roofline = {"bound": "hbm", "kernel": f"m3scan_bwd ({bwd_kernels})",
                "achieved": round(bwd_achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(bwd_achieved / peak, 4), "peak_kind": peak_kind,
                "traffic": ncu_traffic(args.workload, "bwd"),
                "algorithmic_bytes_per_launch": bb,
                "bytes_per_element": round(bb / E, 3),
                "time": "mean call time over the timed steps",
                "median": {"achieved": round(bb / (bwd_med * 1e-3) / 1e9, 1),
                           "frac": round(bb / (bwd_med * 1e-3) / 1e9 / peak, 4)},
                # the path's binding resource: FP32 lane operations
                "alu": {"achieved": round(bwd_gops, 1), "peak": round(alu_peak, 1),
                        "unit": "Gop/s", "frac": round(bwd_gops / alu_peak, 4),
                        "ops_per_element": BWD_FP32_OPS_PER_ELEM,
                        "peak_kind": "derived: 152 SMs x 128 FP32 lanes x max SM clock"}}
    hbm = {"min_bytes_fwd_bwd": fb + bb, "chunk_for_min_bytes": ROOFLINE_CHUNK,
           "frac_of_8TBs": round((fb + bb) / HBM_TARGET_GBS / 1e9 / step_s, 4),
           "frac_of_measured": round((fb + bb) / peak / 1e9 / step_s, 4),
           "fwd_gelem_s": round(E / (fwd_avg * 1e-3) / 1e9, 2),
           "bwd_gelem_s": round(E / (bwd_avg * 1e-3) / 1e9, 2),
           "median": {"ms_per_step": round(step_med, 5),
                      "gelem_s": round(E / (step_med * 1e-3) / 1e9, 3),
                      "fwd_gelem_s": round(E / (fwd_med * 1e-3) / 1e9, 2),
                      "bwd_gelem_s": round(E / (bwd_med * 1e-3) / 1e9, 2),
                      "frac_of_measured": round((fb + bb) / peak / 1e9 / (step_med * 1e-3), 4)}}

    # end to end through the public binding with pinned host buffers
    e2e = None if args.no_e2e else e2e_measure(torch, binding, layer, tensors,
                                               min(args.steps, 50), device)
    if dist is not None and e2e is not None:  # whole-job figures: every replica's elements over the slowest time
        for part in (e2e, e2e["serial"], e2e["eager"]):
            ms = max_over_ranks(dist, part["ms_per_step"], device)
            part["ms_per_step"] = round(ms, 5)
            part["value"] = round(job_gelem_s(world, E, 1, ms), 3)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": w.batch, "seq_len": w.seq_len,
                   "d_inner": w.d_inner, "d_state": NS, "d_conv": 4, "act_storage": w.act,
                   "chunk": int(layer.plan.chunk), "fwd_segments": int(layer.plan.fwd_segments),
                   "bwd_segments": int(layer.plan.bwd_segments),
                   "fwd_launches": int(layer.plan.fwd_launches),
                   "bwd_launches": int(layer.plan.bwd_launches),
                   "l2": "flushed before every step (256 MiB memset, then read back so that no write-back of it is timed; outside the events)",
                   "timing": "CUDA graphs (fwd, bwd) per step, CUDA events per graph",
                   "parallelism": f"replicas x{world}"},
        "hbm_roofline": hbm,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": int(args.steps * (layer.plan.fwd_launches + layer.plan.bwd_launches)),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
    if rank == 0 and not args.no_extras:
        line["extra"] = extras(torch, binding, device, args, flush, stream)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def _packed(torch, shapes, device, pin):
    """One buffer holding every tensor of ``shapes`` (name -> (shape, dtype))
    at 256-byte aligned offsets, and a view per name."""
    offs, off = {}, 0
    for k, (shape, dt) in shapes.items():
        offs[k] = off
        n = int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
        off = (off + n + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=device, pin_memory=pin)
    views = {}
    for k, (shape, dt) in shapes.items():
        n = int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
        views[k] = buf[offs[k]:offs[k] + n].view(dt).view(shape)
    return buf, views


def e2e_measure(torch, binding, layer, tensors, steps, device):
    """Same step through the public binding, with the step's inputs copied
    from pinned host memory and its results copied back inside the events.
    The inputs sit in one pinned host buffer (as a data loader would hand
    over a batch) and the outputs come back into one, so a step is one
    host-to-device copy, the forward and backward, and one device-to-host
    copy.  Reported two ways: the step captured once as a CUDA graph and
    replayed -- how a loop over small layers runs -- and the same calls
    issued eagerly from Python every step."""
    ins = ("x", "delta_raw", "z", "B", "C", "d_gated", "conv_w", "conv_b", "dt_bias",
           "a_log", "D")
    outs = ("gated", "d_x", "d_delta_raw", "dz", "dB", "dC", "d_conv_w", "d_conv_b",
            "d_dt_bias", "d_a_log", "dD")
    in_shapes = {k: (tuple(tensors[k].shape), tensors[k].dtype) for k in ins}
    out_shapes = {k: (tuple(layer.o[k].shape), layer.o[k].dtype) for k in outs}
    h_in_buf, h_in = _packed(torch, in_shapes, "cpu", True)
    d_in_buf, d_in = _packed(torch, in_shapes, device, False)
    h_out_buf, _ = _packed(torch, out_shapes, "cpu", True)
    d_out_buf, d_out = _packed(torch, out_shapes, device, False)
    for k in ins:
        h_in[k].copy_(tensors[k].cpu())
    bi = h_in_buf.numel()
    bo = h_out_buf.numel()
    ws = layer.ws
    E = layer.shape[0] * layer.shape[1] * layer.shape[2]

    def step(s):
        d_in_buf.copy_(h_in_buf, non_blocking=True)
        binding.m3scan_fwd(
            d_in["x"], d_in["delta_raw"], d_in["z"], d_in["B"], d_in["C"], d_in["conv_w"],
            d_in["conv_b"], d_in["dt_bias"], d_in["a_log"], d_in["D"], chunk=int(layer.plan.chunk),
            segments=layer.segments, threads_per_channel=layer.tpc,
            gated=d_out["gated"], ckpt=layer.o["ckpt"], workspace=_WS(ws), stream=s)
        binding.m3scan_bwd(
            d_in["x"], d_in["delta_raw"], d_in["z"], d_in["B"], d_in["C"], d_in["conv_w"],
            d_in["conv_b"], d_in["dt_bias"], d_in["a_log"], d_in["D"], layer.o["ckpt"],
            d_in["d_gated"], chunk=int(layer.plan.chunk), segments=layer.segments,
            threads_per_channel=layer.tpc, deterministic=layer.deterministic,
            out={k: d_out[k] for k in outs if k != "gated"}, workspace=_WS(ws), stream=s)
        h_out_buf.copy_(d_out_buf, non_blocking=True)

    def timed(run):
        s = torch.cuda.current_stream()
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            run()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_eager = timed(lambda: step(torch.cuda.current_stream()))
    side = torch.cuda.Stream(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        step(side)  # warm the plan cache on the capture stream
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        step(side)
    ms_serial = timed(graph.replay)

    # Pipelined: a copy-in stream, the compute stream and a copy-out stream,
    # with the device input and output buffers doubled, so step k+1's inputs
    # arrive and step k-1's results leave while step k computes (a data
    # loader's prefetch).  Every step still copies its own inputs in and its
    # own results out.  Captured as one graph of `depth` steps and replayed.
    depth = 10
    d_in2 = [(d_in_buf, d_in), _packed(torch, in_shapes, device, False)]
    d_out2 = [(d_out_buf, d_out), _packed(torch, out_shapes, device, False)]
    sh, sd = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def pipe(sc, n):
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()]
              for k in ("in_ready", "in_free", "out_ready", "out_free")}
        sh.wait_stream(sc)
        sd.wait_stream(sc)
        for k in range(n):
            b = k % 2
            dib, di = d_in2[b]
            dob, do = d_out2[b]
            if k >= 2:
                sh.wait_event(ev["in_free"][b])
            with torch.cuda.stream(sh):
                dib.copy_(h_in_buf, non_blocking=True)
            ev["in_ready"][b].record(sh)
            sc.wait_event(ev["in_ready"][b])
            if k >= 2:
                sc.wait_event(ev["out_free"][b])
            binding.m3scan_fwd(
                di["x"], di["delta_raw"], di["z"], di["B"], di["C"], di["conv_w"],
                di["conv_b"], di["dt_bias"], di["a_log"], di["D"], chunk=int(layer.plan.chunk),
                segments=layer.segments, threads_per_channel=layer.tpc,
                gated=do["gated"], ckpt=layer.o["ckpt"], workspace=_WS(ws), stream=sc)
            binding.m3scan_bwd(
                di["x"], di["delta_raw"], di["z"], di["B"], di["C"], di["conv_w"],
                di["conv_b"], di["dt_bias"], di["a_log"], di["D"], layer.o["ckpt"],
                di["d_gated"], chunk=int(layer.plan.chunk), segments=layer.segments,
                threads_per_channel=layer.tpc, deterministic=layer.deterministic,
                out={k2: do[k2] for k2 in outs if k2 != "gated"}, workspace=_WS(ws), stream=sc)
            ev["in_free"][b].record(sc)
            ev["out_ready"][b].record(sc)
            sd.wait_event(ev["out_ready"][b])
            with torch.cuda.stream(sd):
                h_out_buf.copy_(dob, non_blocking=True)
            ev["out_free"][b].record(sd)
        sc.wait_stream(sh)
        sc.wait_stream(sd)

    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        pipe(side, 2)
    torch.cuda.synchronize()
    with torch.cuda.graph(pgraph, stream=side):
        pipe(side, depth)
    ms = timed(pgraph.replay) / depth
    return {"value": round(E / (ms * 1e-3) / 1e9, 3), "unit": UNIT,
            "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
            "ms_per_step": round(ms, 5), "steps": steps * depth,
            "how": "inputs in one pinned host buffer copied in, fwd + bwd through the binding, "
                   "all outputs copied back into one pinned buffer; copies in and out on their "
                   "own streams with doubled device buffers, so they overlap the neighbouring "
                   "steps' compute; captured as one CUDA graph of 10 steps and replayed",
            "serial": {"value": round(E / (ms_serial * 1e-3) / 1e9, 3),
                       "ms_per_step": round(ms_serial, 5),
                       "how": "copy in, fwd + bwd, copy out on one stream, the step captured as a "
                              "CUDA graph and replayed"},
            "eager": {"value": round(E / (ms_eager * 1e-3) / 1e9, 3),
                      "ms_per_step": round(ms_eager, 5),
                      "how": "the serial step's calls issued from Python every step"}}


class _WS:
    def __init__(self, buf):
        self.buf = buf
        self.nbytes = buf.numel()
        self.ptr = buf.data_ptr()


def extras(torch, binding, device, args, flush, stream):
    """The larger workloads at full size (device-drawn inputs, same recipe
    distributions), and the 24-layer stack of the Mamba-2.8B-like core."""
    out = {}
    for name in EXTRA_WORKLOADS:
        w = WORKLOADS[name]
        es = 2 if w.act == "bf16" else 4
        t = device_inputs(torch, w, device)
        L = Layer(torch, binding, t)
        with torch.cuda.stream(stream):
            for _ in range(2):
                L.fwd(stream.cuda_stream)
                L.bwd(stream.cuda_stream)
        torch.cuda.synchronize()
        gf, gb = capture(torch, [L], stream)
        for _ in range(2):
            gf.replay()
            gb.replay()
        f_ms, b_ms = time_steps(torch, gf, gb, args.extra_steps, flush)
        fa, ba = sum(f_ms) / len(f_ms), sum(b_ms) / len(b_ms)
        fb, bb = algorithmic_bytes(w.batch, w.seq_len, w.d_inner, es)
        E = w.elems
        out[name] = {"gelem_s": round(E / ((fa + ba) * 1e-3) / 1e9, 2),
                     "fwd_gelem_s": round(E / (fa * 1e-3) / 1e9, 2),
                     "bwd_gelem_s": round(E / (ba * 1e-3) / 1e9, 2),
                     "ms_fwd": round(fa, 4), "ms_bwd": round(ba, 4),
                     "frac_of_8TBs": round((fb + bb) / HBM_TARGET_GBS / 1e9 / ((fa + ba) * 1e-3), 4),
                     "fwd_segments": int(L.plan.fwd_segments),
                     "bwd_segments": int(L.plan.bwd_segments), "chunk": int(L.plan.chunk)}
        if (fb + bb) < L2_BYTES // 4:
            # a step whose data fits in L2 several times over: also timed with
            # the previous step's lines left in L2, as a training loop over
            # such small layers runs it
            wf, wb = time_steps(torch, gf, gb, args.extra_steps, None)
            wfa, wba = sum(wf) / len(wf), sum(wb) / len(wb)
            out[name]["warm_l2"] = {"gelem_s": round(E / ((wfa + wba) * 1e-3) / 1e9, 2),
                                    "fwd_gelem_s": round(E / (wfa * 1e-3) / 1e9, 2),
                                    "bwd_gelem_s": round(E / (wba * 1e-3) / 1e9, 2)}
        del gf, gb, L, t
        torch.cuda.empty_cache()
    if not args.no_stack:
        out["m2p8b_stack24"] = stack24(torch, binding, device, args, stream)
    out["decode"] = decode_extras(torch, binding, device, flush)
    out["conv_bwd"] = conv_bwd_extras(torch, binding, device, flush)
    out["dt_proj"] = dt_proj_extras(torch, device, flush)
    return out


def dt_proj_extras(torch, device, flush, steps=20):
    """The low-rank dt_proj that feeds delta_raw (delta_raw = dt_low W_dt^T,
    dt_rank = d_model / 16), as the unfused path runs it: one bf16 GEMM
    (cuBLAS) writing delta_raw, L2 flushed before each.  Beside it the
    least a fold into the scan kernels would add to the forward alone:
    dt_rank FP32 multiply-adds per element at the GPU's FP32 lane rate (152
    SMs x 128 lanes x the maximum clock), on kernels already bound by
    instruction issue."""
    out = {}
    for name in ("trainer_b8_t128_d512", "m130m_b8_t2048_d1536", "longseq_b1_t65536_d2048",
                 "m2p8b_b4_t4096_d5120"):
        w = WORKLOADS[name]
        R = (w.d_inner // 2 + 15) // 16  # d_model = d_inner / 2
        g = torch.Generator(device=device)
        g.manual_seed(7)
        low = torch.randn(w.batch * w.seq_len, R, device=device, generator=g).to(torch.bfloat16)
        W = (torch.randn(R, w.d_inner, device=device, generator=g) * 0.1).to(torch.bfloat16)
        dr = torch.empty(w.batch * w.seq_len, w.d_inner, device=device, dtype=torch.bfloat16)
        s = torch.cuda.current_stream()
        for _ in range(3):
            torch.matmul(low, W, out=dr)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e0, e1 in ev:
            flush_l2(torch, flush)
            e0.record(s)
            torch.matmul(low, W, out=dr)
            e1.record(s)
        torch.cuda.synchronize()
        ms = sorted(e0.elapsed_time(e1) for e0, e1 in ev)[steps // 2]
        fold_ms = R * w.elems / (alu_peak_gops() * 1e9) * 1e3
        out[name] = {"dt_rank": R, "gemm_us": round(ms * 1e3, 1),
                     "fold_fwd_floor_us": round(fold_ms * 1e3, 1)}
        del low, W, dr
        torch.cuda.empty_cache()
    return out


# one-token decode (m3scan_decode): batch 64 sequences of the Mamba-2.8B-like
# layer (d_inner 5120), bf16 activations, d_state 16, 32 and 64
DECODE_CONFIGS = ((64, 5120, 16), (64, 5120, 32), (64, 5120, 64))


def decode_bytes(B, D, N, es):
    """Bytes one decode step must move: the f32 state read and written, the
    conv state read and written, x, delta_raw, z read and gated written, B and
    C, and the per-channel parameters once."""
    return B * D * (2 * 4 * N + 2 * 3 * es + 4 * es) + 2 * B * N * es + D * (4 * N + 4 * 4 + 3 * 4)


def decode_extras(torch, binding, device, flush, steps=20):
    out = {}
    for (B, D, N) in DECODE_CONFIGS:
        g = torch.Generator(device=device)
        g.manual_seed(1000 + N)
        bf = torch.bfloat16
        rn = lambda *shape, dt=bf: torch.randn(*shape, device=device, generator=g).to(dt)
        x, z = rn(B, 1, D), rn(B, 1, D)
        dr = (0.5 * torch.randn(B, 1, D, device=device, generator=g)).to(bf)
        Bm, Cm = rn(B, 1, N), rn(B, 1, N)
        cw = torch.rand(D, 4, device=device, generator=g) - 0.5
        cb = torch.zeros(D, device=device)
        u = torch.rand(D, device=device, generator=g) * 0.099 + 0.001
        dtb = torch.log(torch.expm1(u))
        alog = torch.log(torch.arange(1, N + 1, device=device, dtype=torch.float32)).repeat(D, 1)
        Dp = torch.ones(D, device=device)
        h = rn(B, N, D, dt=torch.float32)
        c = rn(B, 3, D)
        gated = torch.empty_like(x)
        dims = binding.make_dims(B, 1, D, d_state=N)
        s = torch.cuda.current_stream()
        alog = alog.contiguous()
        args = (dims, binding.M3_BF16, x.data_ptr(), dr.data_ptr(), z.data_ptr(), Bm.data_ptr(),
                Cm.data_ptr(), cw.data_ptr(), cb.data_ptr(), dtb.data_ptr(), alog.data_ptr(),
                Dp.data_ptr(), h.data_ptr(), c.data_ptr(), gated.data_ptr(), None, s.cuda_stream)
        for _ in range(3):
            assert binding.raw_decode(*args) == 0
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e0, e1 in ev:
            flush_l2(torch, flush)
            e0.record(s)
            binding.raw_decode(*args)
            e1.record(s)
        torch.cuda.synchronize()
        ms = sorted(e0.elapsed_time(e1) for e0, e1 in ev)[steps // 2]
        byt = decode_bytes(B, D, N, 2)
        peak, kind = measured_peaks()
        gbs = byt / (ms * 1e-3) / 1e9
        out[f"b{B}_d{D}_n{N}"] = {"us_per_token_step": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                                  "frac_of_hbm": round(gbs / peak, 3), "hbm_peak_kind": kind,
                                  "bytes": int(byt)}
    return out


def conv_bwd_extras(torch, binding, device, flush, steps=20):
    """The second call of the two-phase backward (m3scan_conv_bwd: SiLU and
    conv backward from du plus an extra input gradient) on the large
    workloads: its own launches, L2 flushed before each.  Bytes: x, du and
    du_extra read, d_x written (activation dtype), the parameter partials."""
    out = {}
    for name in ("m130m_b8_t2048_d1536", "m2p8b_b4_t4096_d5120"):
        w = WORKLOADS[name]
        t = device_inputs(torch, w, device)
        Bsz, T, D = t["x"].shape
        es = 2 if w.act == "bf16" else 4
        act = binding.M3_BF16 if es == 2 else binding.M3_F32
        dims = binding.make_dims(Bsz, T, D)
        pl = binding.m3scan_plan(dims, act)
        ws = binding.Workspace(pl.workspace_bytes, device)
        du, due, dx = torch.randn_like(t["x"]), torch.randn_like(t["x"]), torch.empty_like(t["x"])
        dw = torch.empty(D, 4, device=device)
        db = torch.empty(D, device=device)
        s = torch.cuda.current_stream()
        args = (dims, act, t["x"].data_ptr(), t["conv_w"].data_ptr(), t["conv_b"].data_ptr(),
                du.data_ptr(), due.data_ptr(), dx.data_ptr(), dw.data_ptr(), db.data_ptr(), None,
                ws.ptr, ws.nbytes, s.cuda_stream)
        for _ in range(3):
            assert binding.raw_conv_bwd(*args) == 0
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e0, e1 in ev:
            flush_l2(torch, flush)
            e0.record(s)
            binding.raw_conv_bwd(*args)
            e1.record(s)
        torch.cuda.synchronize()
        ms = sorted(e0.elapsed_time(e1) for e0, e1 in ev)[steps // 2]
        byt = Bsz * T * D * 4 * es
        peak, kind = measured_peaks()
        gbs = byt / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 1), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 3),
                     "hbm_peak_kind": kind, "bytes": int(byt)}
        del t, du, due, dx, ws
        torch.cuda.empty_cache()
    return out


def stack24(torch, binding, device, args, stream):
    name = "m2p8b_b4_t4096_d5120"
    w = WORKLOADS[name]
    layers = [Layer(torch, binding, device_inputs(torch, w, device, seed_offset=l))
              for l in range(24)]
    with torch.cuda.stream(stream):
        for L in layers:
            L.fwd(stream.cuda_stream)
        for L in reversed(layers):
            L.bwd(stream.cuda_stream)
    torch.cuda.synchronize()
    gf, gb = capture(torch, layers, stream)
    gf.replay()
    gb.replay()
    torch.cuda.synchronize()
    f_ms, b_ms = time_steps(torch, gf, gb, max(2, args.extra_steps // 4), None)
    fa, ba = sum(f_ms) / len(f_ms), sum(b_ms) / len(b_ms)
    fb, bb = algorithmic_bytes(w.batch, w.seq_len, w.d_inner, 2)
    E = 24 * w.elems
    res = {"gelem_s": round(E / ((fa + ba) * 1e-3) / 1e9, 2), "ms_fwd": round(fa, 3),
           "ms_bwd": round(ba, 3),
           "frac_of_8TBs": round(24 * (fb + bb) / HBM_TARGET_GBS / 1e9 / ((fa + ba) * 1e-3), 4),
           "note": "24 independent layer cores, fwd 0..23 then bwd 23..0, one graph each"}
    del gf, gb, layers
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------

def channel_sample(inp, channels):
    """The workload restricted to its first `channels` channels (all batches
    and steps): every per-channel tensor and parameter sliced, B and C whole.
    Channels are independent recurrences, so the oracle computes these
    channels exactly (dB and dC become their sums over the sample)."""
    import numpy as np
    from mamba_selective_scan_gb300.inputs import Inputs
    per_elem = ("x", "delta_raw", "z", "d_gated")
    per_chan = ("conv_w", "conv_b", "dt_bias", "a_log", "D")
    arrays = {}
    for k, v in inp.arrays.items():
        if k in per_elem:
            arrays[k] = np.ascontiguousarray(v[:, :, :channels])
        elif k in per_chan:
            arrays[k] = np.ascontiguousarray(v[:channels])
        else:
            arrays[k] = v
    return Inputs(inp.batch, inp.seq_len, channels, inp.d_state, inp.d_conv, inp.act, arrays)


def oracle_sample_rate(inp, channels):
    """Time the single-threaded oracle's forward + backward on the first
    `channels` channels (all batches and steps) of the workload; returns
    (elements, s).  The slicing is outside the timed region."""
    import oracle
    sub = channel_sample(inp, channels)
    t0 = time.perf_counter()
    oracle.forward(sub)
    oracle.backward(sub)
    dt = time.perf_counter() - t0
    return inp.batch * inp.seq_len * channels, dt


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def pick_channels(inp, seconds):
    """Channels whose oracle fwd+bwd takes about `seconds` (fixed per-call
    overhead measured separately and excluded from the per-channel cost)."""
    oracle_sample_rate(inp, 1)  # load the library, warm caches
    k = min(8, inp.d_inner)
    _, t1 = oracle_sample_rate(inp, 1)
    _, tk = oracle_sample_rate(inp, k)
    per_chan = max((tk - t1) / max(k - 1, 1), tk / k / 4, 1e-6)
    fixed = max(t1 - per_chan, 0.0)
    ch = int(max(seconds - fixed, 0.0) / per_chan)
    return max(1, min(inp.d_inner, ch)), per_chan


def cpu_baseline(inp, seconds):
    """The float64 oracle on the host cores, on a bounded channel sample of
    the workload: single-threaded (the pinned oracle as it stands), and on
    every core (the same oracle, one block of channels per OpenMP thread)."""
    import oracle
    oracle.build()
    host_cores = os.cpu_count() or 1
    ch1, _ = pick_channels(inp, seconds)
    e1, t1 = oracle_sample_rate(inp, ch1)
    single = {"value": round(e1 / t1 / 1e9, 6), "unit": UNIT, "cores": 1,
              "sample": f"first {ch1} of {inp.d_inner} channels, all batches and steps, "
                        f"fwd+bwd ({t1:.1f} s)"}
    try:
        oracle.build_par()
    except Exception as e:  # no OpenMP on this host: the single-threaded figure only
        return {"value": single["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
                "host_cores": host_cores, "model": cpu_model(),
                "sample": single["sample"] + ", float64 C oracle, single thread",
                "single_thread": single, "all_cores": None, "note": f"all-core driver: {e}"}
    chn = min(inp.d_inner, ch1 * host_cores)
    sub = channel_sample(inp, chn)
    t0 = time.perf_counter()
    _, used = oracle.forward_backward_all_cores(sub, 0)
    tn = time.perf_counter() - t0
    en = inp.batch * inp.seq_len * chn
    return {"value": round(en / tn / 1e9, 6), "unit": UNIT, "cores": used, "kind": "oracle",
            "host_cores": host_cores, "model": cpu_model(),
            "sample": f"first {chn} of {inp.d_inner} channels, all batches and steps, fwd+bwd, "
                      f"float64 C oracle on {used} OpenMP threads, one block of channels each "
                      f"({tn:.1f} s)",
            "single_thread": single,
            "all_cores": {"value": round(en / tn / 1e9, 6), "unit": UNIT, "cores": used}}


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = WORKLOADS[args.workload]
    inp = make_workload_inputs(args.workload)
    total_steps = args.steps + args.warmup
    budget = 90.0 / max(total_steps, 1)
    ch, _ = pick_channels(inp, budget)
    for _ in range(args.warmup):
        oracle_sample_rate(inp, ch)
    times = []
    elems = 0
    for _ in range(args.steps):
        e, dt = oracle_sample_rate(inp, ch)
        times.append(dt)
        elems += e
    tot = sum(times)
    value = elems / tot / 1e9
    sample = (f"first {ch} of {w.d_inner} channels per step, all batches and steps, "
              f"fwd+bwd, float64 C, single thread")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": w.batch, "seq_len": w.seq_len,
                       "d_inner": w.d_inner, "d_state": NS, "d_conv": 4, "act_storage": w.act},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample, "model": cpu_model(),
                             "host_cores": os.cpu_count()},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--segments", type=int, default=0)
    ap.add_argument("--threads-per-channel", type=int, default=0,
                    help="kernel variant (0 = chosen by the plan, 1 or 2)")
    ap.add_argument("--deterministic", action="store_true",
                    help="fixed-order sums for dB, dC and the parameter gradients")
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="leave out the end-to-end measurement (kernel sweeps and profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--decode-only", action="store_true",
                    help="run only the one-token decode measurements (for profiling)")
    ap.add_argument("--conv-only", action="store_true",
                    help="run only the two-phase conv-backward measurements (for profiling)")
    ap.add_argument("--write-traffic", metavar="LAUNCHES_CSV",
                    help="write profiles/ncu_traffic.json for --workload from an ncu launch list "
                         "taken on the current kernel code (no GPU needed), then exit")
    args = ap.parse_args()
    if args.write_traffic:
        rec = traffic_from_launch_list(args.write_traffic, args.workload)
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json"), "w") as f:
            json.dump(rec, f, indent=1)
        print(json.dumps(rec["traffic"]))
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.decode_only:
        import torch
        from mamba_selective_scan_gb300 import binding, build
        build.build()
        dev = torch.device("cuda", 0)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        print(json.dumps({"decode": decode_extras(torch, binding, dev, flush, steps=args.steps)}))
        return
    if args.conv_only:
        import torch
        from mamba_selective_scan_gb300 import binding, build
        build.build()
        dev = torch.device("cuda", 0)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        print(json.dumps({"conv_bwd": conv_bwd_extras(torch, binding, dev, flush, steps=args.steps)}))
        return
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()

"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, run the oracle on the same (rounded) inputs, compare.

Error measure: max_i |gpu_i - ref_i| / max_i |ref_i| per output tensor.
Tolerances: float32 activations 1e-4 on every output; bf16 activations with
f32 state 2e-2 on the per-element activation outputs and 5e-3 on the f32
reductions (dB, dC and the parameter gradients).
"""

from __future__ import annotations

import numpy as np

import oracle
from mamba_selective_scan_gb300 import binding
from mamba_selective_scan_gb300.inputs import bf16_bits

ACT_OUT = ("gated", "y", "du", "dz", "d_x", "d_delta_raw")
RED_OUT = ("dB", "dC", "d_a_log", "dD", "d_dt_bias", "d_conv_w", "d_conv_b")
TOL = {
    "f32": {k: 1e-4 for k in ACT_OUT + RED_OUT},
    "bf16": {**{k: 2e-2 for k in ACT_OUT}, **{k: 5e-3 for k in RED_OUT}},
}


def to_device(inp, device="cuda:0"):
    import torch
    out = {}
    for k, v in inp.arrays.items():
        if k in ("x", "delta_raw", "z", "B", "C", "d_gated") and inp.act == "bf16":
            out[k] = torch.from_numpy(bf16_bits(v).view(np.int16)).view(torch.bfloat16).to(device)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(device)
    return out


def to_np(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def run_gpu(dev, chunk=0, segments=0, want_debug=True, d_gated=None, fwd_segments=None, tpc=0,
            det=False):
    """Forward then backward through the C ABI.  Returns dict of float64 arrays."""
    import torch
    seg_f = segments if fwd_segments is None else fwd_segments
    gated, ckpt, y = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                        dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                        dev["a_log"], dev["D"], chunk=chunk, segments=seg_f,
                                        want_y=want_debug, threads_per_channel=tpc)
    g = dev["d_gated"] if d_gated is None else d_gated
    grads = binding.m3scan_bwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                               dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"],
                               dev["D"], ckpt, g, chunk=chunk, segments=segments,
                               want_du=want_debug, threads_per_channel=tpc,
                               deterministic=det)
    torch.cuda.synchronize()
    res = {"gated": to_np(gated), "ckpt": to_np(ckpt)}
    if y is not None:
        res["y"] = to_np(y)
    for k, v in grads.items():
        res[k] = to_np(v)
    return res


def run_oracle(inp, chan_mask=None, d_gated=None):
    f = oracle.forward(inp, chan_mask=chan_mask)
    b = oracle.backward(inp, d_gated=d_gated, chan_mask=chan_mask)
    res = {"gated": f["gated"], "y": f["y"]}
    res.update(b)
    return res


def norm_err(a, ref):
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    diff = float(np.max(np.abs(a - ref))) if ref.size else 0.0
    if scale == 0.0:
        return diff
    return diff / scale


def compare(gpu, ref, act, keys=None, select=None):
    """Return {name: (err, tol)} for every compared output; select(name, arr)
    may slice both sides (e.g. to sampled channels)."""
    tol = TOL[act]
    out = {}
    for k in keys or tol:
        if k not in gpu or k not in ref:
            continue
        a, r = gpu[k], ref[k]
        if select is not None:
            a, r = select(k, a), select(k, r)
        out[k] = (norm_err(a, r), tol[k])
    return out


def assert_close(report, ctx=""):
    bad = {k: v for k, v in report.items() if not v[0] <= v[1]}
    assert not bad, f"{ctx} parity failures (err, tol): {bad}; all: {report}"

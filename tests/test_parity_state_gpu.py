"""GPU parity of the carried-state entry points (m3scan_fwd_state,
m3scan_bwd_state) against the float64 oracle on the same seeded inputs.

Cases cover several chunks, time segments and channel groups, chunks of one
and two steps (whose conv halos reach into the carried conv inputs past the
first chunk), windows shorter than the conv, the empty window, window
chaining on the GPU, and NULL state pointers (which must give the plain
entry points' results bit for bit).
"""

import numpy as np
import pytest

import oracle
from mamba_selective_scan_gb300 import binding
from mamba_selective_scan_gb300.inputs import bf16_bits, make_inputs, make_state_inputs
from parity_util import TOL, assert_close, compare, norm_err, to_device, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# state outputs: the SSM state is an f32 reduction-like quantity, the conv
# state a copy of inputs (exact)
STATE_TOL = {"f32": {"ssm_state_out": 1e-4, "d_ssm_state": 1e-4, "d_conv_state": 1e-4},
             "bf16": {"ssm_state_out": 5e-3, "d_ssm_state": 5e-3, "d_conv_state": 2e-2}}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_selective_scan_gb300 import build
    build.build()


def _state_to_device(st, act):
    out = {}
    for k, v in st.items():
        if k in ("conv_state", "d_conv_state_out") and act == "bf16":
            out[k] = torch.from_numpy(bf16_bits(v).view(np.int16)).view(torch.bfloat16).cuda()
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()
    return out


def _gpu(dev, sd, chunk, segments, use=("ssm_state", "conv_state", "d_ssm_state_out",
                                         "d_conv_state_out"), tpc=0):
    s = {k: (sd[k] if k in use else None) for k in sd}
    gated, ckpt, y, h_out, c_out = binding.m3scan_fwd_state(
        dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"], dev["conv_b"],
        dev["dt_bias"], dev["a_log"], dev["D"], ssm_state=s["ssm_state"],
        conv_state=s["conv_state"], chunk=chunk, segments=segments, want_y=True,
        threads_per_channel=tpc)
    g = binding.m3scan_bwd_state(
        dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"], dev["conv_b"],
        dev["dt_bias"], dev["a_log"], dev["D"], ckpt, dev["d_gated"], conv_state=s["conv_state"],
        d_ssm_state_out=s["d_ssm_state_out"], d_conv_state_out=s["d_conv_state_out"],
        chunk=chunk, segments=segments, want_du=True, threads_per_channel=tpc)
    torch.cuda.synchronize()
    res = {"gated": to_np(gated), "y": to_np(y), "ssm_state_out": to_np(h_out),
           "conv_state_out": to_np(c_out), "ckpt": to_np(ckpt)}
    res.update({k: to_np(v) for k, v in g.items()})
    return res


def _oracle(inp, st, use):
    s = {k: (st[k] if k in use else None) for k in st}
    f = oracle.forward(inp, ssm_state=s["ssm_state"], conv_state=s["conv_state"])
    b = oracle.backward(inp, **s)
    res = dict(b)
    res.update(gated=f["gated"], y=f["y"], ssm_state_out=f["ssm_state_out"],
               conv_state_out=f["conv_state_out"])
    return res


def _check(gpu, ref, act, ctx):
    rep = compare(gpu, ref, act)
    for k, tol in STATE_TOL[act].items():
        rep[k] = (norm_err(gpu[k], ref[k]), tol)
    assert_close(rep, ctx)
    assert np.array_equal(gpu["conv_state_out"], ref["conv_state_out"]), ctx


ALL = ("ssm_state", "conv_state", "d_ssm_state_out", "d_conv_state_out")

CASES = [
    # batch, T, D, act, chunk, segments
    (2, 200, 136, "f32", 16, 3),
    (2, 200, 136, "bf16", 8, 0),
    (2, 97, 72, "bf16", 32, 2),
    (1, 300, 40, "f32", 64, 2),
    (1, 130, 200, "f32", 7, 5),
    (3, 40, 24, "f32", 1, 4),     # one-step chunks: halos of chunks 1, 2 reach the carried inputs
    (2, 41, 40, "bf16", 2, 3),    # two-step chunks
    (1, 2, 8, "f32", 0, 0),       # window shorter than the conv
    (2, 1, 16, "bf16", 1, 0),
    (1, 3, 8, "f32", 2, 0),
    (4, 33, 520, "bf16", 16, 2),
]


@pytest.mark.parametrize("tpc", [1, 2])
@pytest.mark.parametrize("batch,T,D,act,chunk,segments", CASES)
def test_state_in_and_out_match_oracle(batch, T, D, act, chunk, segments, tpc):
    seed = 7 * batch + T + D
    inp = make_inputs(batch, T, D, act=act, seed=seed)
    st = make_state_inputs(batch, D, act=act, seed=seed)
    gpu = _gpu(to_device(inp), _state_to_device(st, act), chunk, segments, tpc=tpc)
    ref = _oracle(inp, st, ALL)
    _check(gpu, ref, act, f"B{batch} T{T} D{D} {act} K{chunk} S{segments} tpc{tpc}")
    assert np.array_equal(gpu["ckpt"][:, 0], st["ssm_state"])


@pytest.mark.parametrize("use", [("ssm_state",), ("conv_state",), ("d_ssm_state_out",),
                                 ("d_conv_state_out",)])
def test_each_state_argument_alone(use):
    batch, T, D, act = 2, 60, 72, "f32"
    inp = make_inputs(batch, T, D, act=act, seed=11)
    st = make_state_inputs(batch, D, act=act, seed=11)
    gpu = _gpu(to_device(inp), _state_to_device(st, act), 4, 3, use=use)
    ref = _oracle(inp, st, use)
    _check(gpu, ref, act, f"only {use}")


def test_null_state_matches_plain_entry_points_bit_for_bit():
    batch, T, D, act = 2, 150, 136, "bf16"
    inp = make_inputs(batch, T, D, act=act, seed=12)
    dev = to_device(inp)
    sd = _state_to_device(make_state_inputs(batch, D, act=act, seed=12), act)
    a = _gpu(dev, sd, 8, 3, use=())
    gated, ckpt, y = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                        dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                        dev["a_log"], dev["D"], chunk=8, segments=3, want_y=True)
    g = binding.m3scan_bwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                           dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"],
                           ckpt, dev["d_gated"], chunk=8, segments=3, want_du=True)
    torch.cuda.synchronize()
    assert np.array_equal(a["gated"], to_np(gated))
    # dB, dC and (split kernel over several segments) the parameter
    # gradients are sums of float atomics: their order may differ between runs
    for k in ("d_x", "d_delta_raw", "dz", "du"):
        assert np.array_equal(a[k], to_np(g[k])), k
    for k in ("dB", "dC", "d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert norm_err(a[k], to_np(g[k])) <= 1e-6, k


def test_empty_window_passes_state_through():
    batch, D, act = 2, 40, "bf16"
    inp = make_inputs(batch, 0, D, act=act, seed=13)
    st = make_state_inputs(batch, D, act=act, seed=13)
    gpu = _gpu(to_device(inp), _state_to_device(st, act), 0, 0)
    assert np.array_equal(gpu["ssm_state_out"], st["ssm_state"])
    assert np.array_equal(gpu["conv_state_out"], st["conv_state"])
    assert np.array_equal(gpu["d_ssm_state"], st["d_ssm_state_out"])
    assert np.array_equal(gpu["d_conv_state"], st["d_conv_state_out"])


def test_two_gpu_windows_equal_one_gpu_window():
    """Forward window 1 then window 2 from its state; backward window 2 then
    window 1 with window 2's state gradients upstream: the same results as
    one call over the whole sequence (within f32 rounding)."""
    batch, T, T1, D, act = 2, 180, 77, 136, "f32"
    inp = make_inputs(batch, T, D, act=act, seed=14)
    st = make_state_inputs(batch, D, act=act, seed=14)
    dev = to_device(inp)
    sd = _state_to_device(st, act)
    full = _gpu(dev, sd, 8, 0)

    def part(t0, t1):
        return {k: (v[:, t0:t1].contiguous() if k in ("x", "delta_raw", "z", "B", "C",
                                                      "d_gated") else v)
                for k, v in dev.items()}

    d1, d2 = part(0, T1), part(T1, T)
    common = lambda d: (d["x"], d["delta_raw"], d["z"], d["B"], d["C"], d["conv_w"],
                        d["conv_b"], d["dt_bias"], d["a_log"], d["D"])
    g1, ck1, _, h1, c1 = binding.m3scan_fwd_state(*common(d1), ssm_state=sd["ssm_state"],
                                                  conv_state=sd["conv_state"], chunk=8)
    g2, ck2, _, h2, c2 = binding.m3scan_fwd_state(*common(d2), ssm_state=h1, conv_state=c1,
                                                  chunk=8)
    b2 = binding.m3scan_bwd_state(*common(d2), ck2, d2["d_gated"], conv_state=c1,
                                  d_ssm_state_out=sd["d_ssm_state_out"],
                                  d_conv_state_out=sd["d_conv_state_out"], chunk=8, want_du=True)
    b1 = binding.m3scan_bwd_state(*common(d1), ck1, d1["d_gated"], conv_state=sd["conv_state"],
                                  d_ssm_state_out=b2["d_ssm_state"],
                                  d_conv_state_out=b2["d_conv_state"], chunk=8, want_du=True)
    torch.cuda.synchronize()
    tol = TOL[act]
    got = np.concatenate([to_np(g1), to_np(g2)], axis=1)
    assert norm_err(got, full["gated"]) <= tol["gated"]
    assert norm_err(to_np(h2), full["ssm_state_out"]) <= 1e-4
    assert np.array_equal(to_np(c2), full["conv_state_out"])
    for k in ("d_x", "d_delta_raw", "dz", "du", "dB", "dC"):
        got = np.concatenate([to_np(b1[k]), to_np(b2[k])], axis=1)
        assert norm_err(got, full[k]) <= tol[k], k
    for k in ("d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert norm_err(to_np(b1[k]) + to_np(b2[k]), full[k]) <= tol[k], k
    for k in ("d_ssm_state", "d_conv_state"):
        assert norm_err(to_np(b1[k]), full[k]) <= 1e-4, k


@pytest.mark.parametrize("N", [32, 64])
def test_wider_state_windows_match_oracle(N):
    batch, T, D, act = 2, 50, 40, "bf16"
    inp = make_inputs(batch, T, D, act=act, seed=N, d_state=N)
    st = make_state_inputs(batch, D, act=act, seed=N, d_state=N)
    gpu = _gpu(to_device(inp), _state_to_device(st, act), 8, 3)
    ref = _oracle(inp, st, ALL)
    _check(gpu, ref, act, f"N={N}")

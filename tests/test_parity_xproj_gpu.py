"""GPU parity of the x_proj neighbours of the layer core.

* Row strides: Bm and Cm as column views of one x_proj output
  [batch, T, dt_rank + 2 d_state] and dB, dC as column views of its f32
  gradient, with no copies; the gradient's other columns stay untouched.
* The two-phase backward (m3scan_bwd_scan, then m3scan_conv_bwd with a
  gradient reaching u from the x_proj path) against the oracle's
  ``d_u_extra``; with no extra gradient it equals the one-call backward.
"""

import numpy as np
import pytest

import oracle
from mamba_selective_scan_gb300 import binding
from mamba_selective_scan_gb300.inputs import bf16_bits, make_inputs, make_state_inputs
from parity_util import TOL, norm_err, to_device, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_selective_scan_gb300 import build
    build.build()


def _act(v, act):
    if act == "bf16":
        return torch.from_numpy(bf16_bits(v).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()


@pytest.mark.parametrize("act,R,segments", [("bf16", 16, 3), ("f32", 48, 1), ("bf16", 160, 0)])
def test_strided_b_c_and_gradients_match_oracle(act, R, segments):
    batch, T, D, N = 2, 150, 136, 16
    inp = make_inputs(batch, T, D, act=act, seed=R + segments)
    dev = to_device(inp)
    L = R + 2 * N
    # x_proj output with B and C in its last 2N columns; dt_low columns hold noise
    xdbl = torch.randn(batch, T, L, device="cuda").to(dev["x"].dtype)
    xdbl[..., R:R + N] = dev["B"]
    xdbl[..., R + N:] = dev["C"]
    Bv, Cv = xdbl[..., R:R + N], xdbl[..., R + N:]
    gdbl = torch.full((batch, T, L), 7.0, device="cuda")  # sentinel in the dt_low columns
    dBv, dCv = gdbl[..., R:R + N], gdbl[..., R + N:]
    dims = binding.make_dims(batch, T, D, chunk=8, segments=segments, bc_stride=L, dbc_stride=L)
    code = binding.M3_BF16 if act == "bf16" else binding.M3_F32
    pl = binding.m3scan_plan(dims, code)
    ws = binding.Workspace(pl.workspace_bytes, dev["x"].device)
    gated = torch.empty_like(dev["x"])
    ckpt = torch.empty((batch, pl.n_chunks, N, D), device="cuda")
    P = lambda k: dev[k].data_ptr()
    st = binding.raw_fwd(dims, code, P("x"), P("delta_raw"), P("z"), Bv.data_ptr(), Cv.data_ptr(),
                         P("conv_w"), P("conv_b"), P("dt_bias"), P("a_log"), P("D"),
                         gated.data_ptr(), None, ckpt.data_ptr(), ws.ptr, ws.nbytes, None)
    assert st == 0, binding.m3scan_status_string(st)
    g = {k: torch.empty_like(dev["x"]) for k in ("d_x", "d_delta_raw", "dz")}
    f = {k: torch.zeros(s, device="cuda") for k, s in
         (("d_conv_w", (D, 4)), ("d_conv_b", (D,)), ("d_dt_bias", (D,)), ("d_a_log", (D, N)),
          ("dD", (D,)))}
    st = binding.raw_bwd(dims, code, P("x"), P("delta_raw"), P("z"), Bv.data_ptr(), Cv.data_ptr(),
                         P("conv_w"), P("conv_b"), P("dt_bias"), P("a_log"), P("D"),
                         ckpt.data_ptr(), P("d_gated"), g["d_x"].data_ptr(),
                         g["d_delta_raw"].data_ptr(), g["dz"].data_ptr(), None, dBv.data_ptr(),
                         dCv.data_ptr(), f["d_conv_w"].data_ptr(), f["d_conv_b"].data_ptr(),
                         f["d_dt_bias"].data_ptr(), f["d_a_log"].data_ptr(), f["dD"].data_ptr(),
                         ws.ptr, ws.nbytes, None)
    assert st == 0, binding.m3scan_status_string(st)
    torch.cuda.synchronize()
    ref_f = oracle.forward(inp)
    ref_b = oracle.backward(inp)
    tol = TOL[act]
    assert norm_err(to_np(gated), ref_f["gated"]) <= tol["gated"]
    got = {"dB": to_np(dBv), "dC": to_np(dCv), **{k: to_np(v) for k, v in g.items()},
           **{k: to_np(v) for k, v in f.items()}}
    for k, v in got.items():
        assert norm_err(v, ref_b[k]) <= tol[k], k
    assert bool((gdbl[..., :R] == 7.0).all())


@pytest.mark.parametrize("batch,T,D,act,chunk,segments,state", [
    (2, 200, 136, "f32", 16, 3, False),
    (2, 200, 136, "bf16", 8, 0, True),
    (8, 128, 512, "bf16", 0, 0, False),     # trainer shape: 32-step conv tiles
    (1, 2, 8, "f32", 0, 0, True),           # shorter than the conv
    (3, 37, 72, "bf16", 2, 4, True),
])
@pytest.mark.parametrize("tpc", [1, 2])
@pytest.mark.parametrize("det", [False, True])
def test_two_phase_backward_matches_oracle(batch, T, D, act, chunk, segments, state, tpc, det):
    """det: dB/dC as fixed-order sums (m3_dims.deterministic), and a
    second call must repeat every output bit for bit."""
    seed = batch + T + D + chunk
    inp = make_inputs(batch, T, D, act=act, seed=seed)
    dev = to_device(inp)
    rng = np.random.default_rng(seed)
    du_extra = rng.standard_normal((batch, T, D)).astype(np.float32)
    du_extra_t = _act(du_extra, act)
    du_extra_rounded = to_np(du_extra_t)
    kw = {}
    st = None
    if state:
        st = make_state_inputs(batch, D, act=act, seed=seed)
        kw = dict(conv_state=_act(st["conv_state"], act),
                  d_ssm_state_out=torch.from_numpy(st["d_ssm_state_out"]).cuda(),
                  d_conv_state_out=_act(st["d_conv_state_out"], act))
        gated, ckpt, _, _, _ = binding.m3scan_fwd_state(
            dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"],
            dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"],
            ssm_state=torch.from_numpy(st["ssm_state"]).cuda(), conv_state=kw["conv_state"],
            chunk=chunk, segments=segments)
    else:
        gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"],
                                            dev["C"], dev["conv_w"], dev["conv_b"],
                                            dev["dt_bias"], dev["a_log"], dev["D"], chunk=chunk,
                                            segments=segments)
    def run():
        return binding.m3scan_bwd_two_phase(
            dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"],
            dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"], ckpt, dev["d_gated"],
            lambda g: du_extra_t, chunk=chunk, segments=segments, threads_per_channel=tpc,
            deterministic=det, **kw)
    o = run()
    torch.cuda.synchronize()
    if det:
        o2 = run()
        torch.cuda.synchronize()
        for k in o:
            assert np.array_equal(to_np(o[k]), to_np(o2[k])), k
    okw = {}
    if state:
        okw = {k: st[k] for k in ("ssm_state", "conv_state", "d_ssm_state_out",
                                  "d_conv_state_out")}
    ref = oracle.backward(inp, d_u_extra=du_extra_rounded, **okw)
    tol = TOL[act]
    for k in ("du", "dz", "d_delta_raw", "dB", "dC", "d_dt_bias", "d_a_log", "dD", "d_x",
              "d_conv_w", "d_conv_b"):
        err = norm_err(to_np(o[k]), ref[k])
        assert err <= tol[k], (k, err)
    if state:
        for k, t in (("d_ssm_state", 1e-4 if act == "f32" else 5e-3),
                     ("d_conv_state", 1e-4 if act == "f32" else 2e-2)):
            err = norm_err(to_np(o[k]), ref[k])
            assert err <= t, (k, err)


def test_two_phase_without_extra_equals_one_call_backward():
    batch, T, D, act = 2, 160, 136, "f32"
    inp = make_inputs(batch, T, D, act=act, seed=9)
    dev = to_device(inp)
    gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                        dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                        dev["a_log"], dev["D"], chunk=8, segments=4)
    one = binding.m3scan_bwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                             dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"],
                             ckpt, dev["d_gated"], chunk=8, segments=4, want_du=True)
    two = binding.m3scan_bwd_two_phase(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                       dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                       dev["a_log"], dev["D"], ckpt, dev["d_gated"], None,
                                       chunk=8, segments=4)
    torch.cuda.synchronize()
    for k in ("du", "dz", "d_delta_raw"):
        assert torch.equal(one[k], two[k]), k
    # d_x at segment boundaries, dB/dC and the parameter gradients (float
    # atomics) are added in another order
    for k in ("d_x", "dB", "dC", "d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert norm_err(to_np(two[k]), to_np(one[k])) <= 1e-6, k


def test_two_phase_backward_with_wider_state():
    batch, T, D, act, N = 2, 60, 40, "f32", 32
    inp = make_inputs(batch, T, D, act=act, seed=21, d_state=N)
    dev = to_device(inp)
    du_extra = np.random.default_rng(21).standard_normal((batch, T, D)).astype(np.float32)
    gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                        dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                        dev["a_log"], dev["D"], chunk=8, segments=2)
    o = binding.m3scan_bwd_two_phase(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                     dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"],
                                     dev["D"], ckpt, dev["d_gated"], lambda g: _act(du_extra, act),
                                     chunk=8, segments=2)
    torch.cuda.synchronize()
    ref = oracle.backward(inp, d_u_extra=du_extra)
    for k in ("du", "dB", "dC", "d_a_log", "d_x", "d_conv_w"):
        assert norm_err(to_np(o[k]), ref[k]) <= TOL[act][k], k

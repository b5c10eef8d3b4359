"""GPU parity with per-channel parameters that differ from channel to channel.

The recipe's workloads fix a_log[d, n] = log(n + 1) for every channel, conv_b
= 0 and D = 1, so a kernel that read one channel's a_log row for all
channels, dropped conv_b or treated D as 1 would still match the oracle on
them.  Every case here draws those three per channel (``random_params``:
a_log ~ U(-4, 3), so exp(delta A) reaches both nearly 1 and nearly 0; conv_b
~ U(-0.5, 0.5); D ~ U(-1.5, 1.5)) and runs each kernel variant against the
float64 oracle on the same inputs: one and two threads per channel, d_state
16/32/64, one and several time segments, deterministic sums, carried state,
the two-phase backward, decode, the no-allocation backward, and the large
workloads at full size on sampled channels.
"""

import numpy as np
import pytest

import oracle
from mamba_selective_scan_gb300 import binding
from mamba_selective_scan_gb300.inputs import (WORKLOADS, bf16_bits, make_inputs,
                                               make_state_inputs, make_workload_inputs)
from parity_util import (TOL, assert_close, compare, norm_err, run_gpu, run_oracle, to_device,
                         to_np)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_selective_scan_gb300 import build
    build.build()


def _inp(batch, T, D, act, seed, N=16):
    return make_inputs(batch, T, D, act=act, seed=seed, d_state=N, random_params=True)


def _act(v, act):
    if act == "bf16":
        return torch.from_numpy(bf16_bits(v).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()


CASES = [
    # batch, T, D, act, chunk, segments, N
    (1, 64, 32, "f32", 0, 0, 16),
    (2, 200, 136, "f32", 16, 3, 16),
    (2, 200, 136, "bf16", 8, 0, 16),
    (2, 97, 72, "bf16", 5, 4, 16),
    (1, 130, 200, "f32", 7, 5, 16),
    (4, 33, 520, "bf16", 16, 2, 16),
    (1, 200, 64, "bf16", 4, 12, 16),
    (2, 100, 64, "f32", 8, 3, 32),
    (3, 33, 136, "bf16", 0, 0, 32),
    (2, 97, 48, "bf16", 16, 2, 64),
    (1, 40, 24, "f32", 2, 4, 64),
]


@pytest.mark.parametrize("tpc", [1, 2])
@pytest.mark.parametrize("batch,T,D,act,chunk,segments,N", CASES)
def test_random_parameters_match_oracle(batch, T, D, act, chunk, segments, N, tpc):
    if N != 16 and tpc == 1:
        pytest.skip("one thread per channel carries 16 state lanes only")
    inp = _inp(batch, T, D, act, seed=batch * 1000 + T + D + N, N=N)
    gpu = run_gpu(to_device(inp), chunk=chunk, segments=segments, tpc=tpc)
    assert_close(compare(gpu, run_oracle(inp), act),
                 f"random params B={batch} T={T} D={D} {act} K={chunk} S={segments} N={N} tpc={tpc}")


@pytest.mark.parametrize("tpc", [1, 2])
@pytest.mark.parametrize("batch,T,D,act,chunk,segments", [
    (2, 200, 136, "f32", 16, 3),
    (2, 97, 72, "bf16", 8, 6),
])
def test_random_parameters_deterministic_sums(batch, T, D, act, chunk, segments, tpc):
    inp = _inp(batch, T, D, act, seed=batch * 77 + T + D)
    dev = to_device(inp)
    a = run_gpu(dev, chunk=chunk, segments=segments, tpc=tpc, det=True)
    b = run_gpu(dev, chunk=chunk, segments=segments, tpc=tpc, det=True)
    assert_close(compare(a, run_oracle(inp), act), f"deterministic, random params tpc={tpc}")
    for k in a:
        assert np.array_equal(a[k], b[k]), k


STATE_TOL = {"f32": {"ssm_state_out": 1e-4, "d_ssm_state": 1e-4, "d_conv_state": 1e-4},
             "bf16": {"ssm_state_out": 5e-3, "d_ssm_state": 5e-3, "d_conv_state": 2e-2}}


@pytest.mark.parametrize("tpc", [1, 2])
@pytest.mark.parametrize("batch,T,D,act,chunk,segments,N", [
    (2, 200, 136, "f32", 16, 3, 16),
    (2, 41, 40, "bf16", 2, 3, 16),
    (2, 50, 40, "bf16", 8, 3, 64),
])
def test_random_parameters_carried_state(batch, T, D, act, chunk, segments, N, tpc):
    if N != 16 and tpc == 1:
        pytest.skip("one thread per channel carries 16 state lanes only")
    seed = 7 * batch + T + D
    inp = _inp(batch, T, D, act, seed=seed, N=N)
    st = make_state_inputs(batch, D, act=act, seed=seed, d_state=N)
    dev = to_device(inp)
    h0 = torch.from_numpy(st["ssm_state"]).cuda()
    c0 = _act(st["conv_state"], act)
    gh = torch.from_numpy(st["d_ssm_state_out"]).cuda()
    gc = _act(st["d_conv_state_out"], act)
    common = (dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"],
              dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"])
    gated, ckpt, y, h_out, c_out = binding.m3scan_fwd_state(
        *common, ssm_state=h0, conv_state=c0, chunk=chunk, segments=segments, want_y=True,
        threads_per_channel=tpc)
    g = binding.m3scan_bwd_state(*common, ckpt, dev["d_gated"], conv_state=c0,
                                 d_ssm_state_out=gh, d_conv_state_out=gc, chunk=chunk,
                                 segments=segments, want_du=True, threads_per_channel=tpc)
    torch.cuda.synchronize()
    got = {"gated": to_np(gated), "y": to_np(y), "ssm_state_out": to_np(h_out)}
    got.update({k: to_np(v) for k, v in g.items()})
    f = oracle.forward(inp, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    ref = oracle.backward(inp, **st)
    ref.update(gated=f["gated"], y=f["y"], ssm_state_out=f["ssm_state_out"])
    rep = compare(got, ref, act)
    for k, tol in STATE_TOL[act].items():
        rep[k] = (norm_err(got[k], ref[k]), tol)
    assert_close(rep, f"carried state, random params N={N} tpc={tpc}")
    assert np.array_equal(to_np(c_out), f["conv_state_out"])


@pytest.mark.parametrize("act,tpc,det", [("bf16", 1, False), ("f32", 2, False), ("bf16", 2, True)])
def test_random_parameters_two_phase_backward(act, tpc, det):
    batch, T, D, chunk, segments = 2, 150, 136, 8, 3
    inp = _inp(batch, T, D, act, seed=33 + tpc)
    dev = to_device(inp)
    du_extra = np.random.default_rng(33).standard_normal((batch, T, D)).astype(np.float32)
    du_extra_t = _act(du_extra, act)
    gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                        dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                        dev["a_log"], dev["D"], chunk=chunk, segments=segments,
                                        threads_per_channel=tpc)
    o = binding.m3scan_bwd_two_phase(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                     dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"],
                                     dev["D"], ckpt, dev["d_gated"], lambda g: du_extra_t,
                                     chunk=chunk, segments=segments, threads_per_channel=tpc,
                                     deterministic=det)
    torch.cuda.synchronize()
    ref = oracle.backward(inp, d_u_extra=to_np(du_extra_t))
    for k in ("du", "dz", "d_delta_raw", "dB", "dC", "d_dt_bias", "d_a_log", "dD", "d_x",
              "d_conv_w", "d_conv_b"):
        err = norm_err(to_np(o[k]), ref[k])
        assert err <= TOL[act][k], (k, err)


@pytest.mark.parametrize("batch,T,D,N,act", [
    (4, 1, 200, 16, "bf16"),
    (2, 5, 136, 32, "f32"),
    (3, 2, 72, 64, "bf16"),
    (65, 1, 520, 16, "f32"),
])
def test_random_parameters_decode(batch, T, D, N, act):
    seed = batch * 100 + T * 10 + N + D
    inp = _inp(batch, T, D, act, seed=seed, N=N)
    st = make_state_inputs(batch, D, act=act, seed=seed, d_state=N)
    dev = to_device(inp)
    h = torch.from_numpy(st["ssm_state"]).cuda()
    c = _act(st["conv_state"], act)
    gated, y = binding.m3scan_decode(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                     dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"],
                                     dev["D"], h, c, want_y=True)
    torch.cuda.synchronize()
    ref = oracle.forward(inp, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    tol = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 5e-3)}[act]
    assert norm_err(to_np(gated), ref["gated"]) <= tol[0]
    assert norm_err(to_np(y), ref["y"]) <= tol[0]
    assert norm_err(to_np(h), ref["ssm_state_out"]) <= tol[1]
    assert np.array_equal(to_np(c), ref["conv_state_out"])


@pytest.mark.parametrize("name", ["m130m_b8_t2048_d1536", "longseq_b1_t65536_d2048",
                                  "m2p8b_b4_t4096_d5120"])
def test_random_parameters_full_size_sampled(name):
    """A large workload at full size in the benchmark's launch configuration
    (library defaults), with per-channel parameters: per-channel outputs and
    parameter gradients on sampled channels, dB/dC with the upstream gradient
    zeroed outside the sample (so the oracle's sampled sums are exact)."""
    w = WORKLOADS[name]
    inp = make_workload_inputs(name, random_params=True)
    dev = to_device(inp)
    D = w.d_inner
    chans = sorted({0, 1, 31, 32, 63, 64, D // 2 + 3, D - 65, D - 1})
    mask = np.zeros(D, dtype=np.uint8)
    mask[chans] = 1
    on = mask.astype(bool)
    gpu = run_gpu(dev)
    ref = run_oracle(inp, chan_mask=mask)

    def sel(k, a):
        if k in ("dB", "dC"):  # [batch, T, d_state]: compared in the second run below
            return a
        return a[:, :, on] if a.ndim == 3 else a[on]
    rep = compare(gpu, ref, w.act, select=sel)
    rep.pop("dB", None)
    rep.pop("dC", None)
    assert_close(rep, name + " random params (sampled channels)")
    gm = inp.arrays["d_gated"] * mask[None, None, :]
    dgm = _act(gm, w.act)
    gpu2 = run_gpu(dev, d_gated=dgm, want_debug=False)
    ref2 = oracle.backward(inp, chan_mask=mask)
    assert_close(compare(gpu2, ref2, w.act, keys=("dB", "dC")), name + " random params (dB/dC)")

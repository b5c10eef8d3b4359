"""GPU parity of m3scan_decode (a short window from the carried state,
updated in place) against the float64 oracle, for d_state 16, 32 and 64,
one-token and multi-token windows, ragged d_inner; and token-by-token decode
against one m3scan_fwd_state call over the same window.
"""

import numpy as np
import pytest

import oracle
from mamba_selective_scan_gb300 import binding
from mamba_selective_scan_gb300.inputs import bf16_bits, make_inputs, make_state_inputs
from parity_util import norm_err, to_device, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = {"f32": {"gated": 1e-4, "y": 1e-4, "ssm_state_out": 1e-4},
       "bf16": {"gated": 2e-2, "y": 2e-2, "ssm_state_out": 5e-3}}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_selective_scan_gb300 import build
    build.build()


def _act_tensor(v, act):
    if act == "bf16":
        return torch.from_numpy(bf16_bits(v).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()


def _decode(dev, h, c, want_y=True):
    return binding.m3scan_decode(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                 dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"],
                                 dev["D"], h, c, want_y=want_y)


CASES = [
    # batch, T, D, N, act
    (4, 1, 200, 16, "bf16"),
    (4, 1, 200, 32, "bf16"),
    (3, 1, 72, 64, "bf16"),
    (2, 1, 136, 16, "f32"),
    (2, 1, 136, 32, "f32"),
    (2, 1, 136, 64, "f32"),
    (2, 5, 130, 16, "f32"),     # multi-token window, d_inner not a multiple of 8
    (2, 7, 72, 64, "bf16"),
    (1, 2, 5, 32, "f32"),       # fewer channels than a warp
    (65, 1, 5120, 16, "bf16"),  # large batch: two rows per thread, odd row count
    (64, 2, 5000, 32, "f32"),   # two rows per thread, ragged channel block
]


@pytest.mark.parametrize("batch,T,D,N,act", CASES)
def test_decode_matches_oracle(batch, T, D, N, act):
    seed = batch * 100 + T * 10 + N + D
    inp = make_inputs(batch, T, D, act=act, seed=seed, d_state=N)
    st = make_state_inputs(batch, D, act=act, seed=seed, d_state=N)
    dev = to_device(inp)
    h = torch.from_numpy(st["ssm_state"]).cuda()
    c = _act_tensor(st["conv_state"], act)
    gated, y = _decode(dev, h, c)
    torch.cuda.synchronize()
    ref = oracle.forward(inp, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    got = {"gated": to_np(gated), "y": to_np(y), "ssm_state_out": to_np(h)}
    for k, tol in TOL[act].items():
        err = norm_err(got[k], ref[k])
        assert err <= tol, (k, err, tol)
    assert np.array_equal(to_np(c), ref["conv_state_out"])


@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_token_by_token_decode_equals_one_state_window(act):
    batch, T, D = 3, 12, 136
    inp = make_inputs(batch, T, D, act=act, seed=5)
    st = make_state_inputs(batch, D, act=act, seed=5)
    dev = to_device(inp)
    h0 = torch.from_numpy(st["ssm_state"]).cuda()
    c0 = _act_tensor(st["conv_state"], act)
    gated_w, _, _, h_w, c_w = binding.m3scan_fwd_state(
        dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"], dev["conv_b"],
        dev["dt_bias"], dev["a_log"], dev["D"], ssm_state=h0, conv_state=c0, chunk=4)
    h, c = h0.clone(), c0.clone()
    outs = []
    for t in range(T):
        one = {k: (v[:, t:t + 1].contiguous() if k in ("x", "delta_raw", "z", "B", "C",
                                                        "d_gated") else v)
               for k, v in dev.items()}
        g, _ = _decode(one, h, c, want_y=False)
        outs.append(g)
    torch.cuda.synchronize()
    tol = TOL[act]
    assert norm_err(to_np(torch.cat(outs, 1)), to_np(gated_w)) <= tol["gated"]
    assert norm_err(to_np(h), to_np(h_w)) <= tol["ssm_state_out"]
    assert torch.equal(c, c_w)


def test_empty_window_leaves_state_unchanged():
    batch, D, act = 2, 64, "bf16"
    inp = make_inputs(batch, 0, D, act=act, seed=6)
    st = make_state_inputs(batch, D, act=act, seed=6)
    dev = to_device(inp)
    h = torch.from_numpy(st["ssm_state"]).cuda()
    c = _act_tensor(st["conv_state"], act)
    h1, c1 = h.clone(), c.clone()
    _decode(dev, h, c, want_y=False)
    torch.cuda.synchronize()
    assert torch.equal(h, h1) and torch.equal(c, c1)

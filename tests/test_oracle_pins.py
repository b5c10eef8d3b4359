"""Pins for the CPU oracle: each test checks it against something other than
itself -- finite differences, closed forms, library routines
(numpy.convolve, scipy.signal.lfilter, torch autograd), brute-force sums and
invariants that the layer core's equations fix.

The equations pinned are those of the Mamba-1 selective-scan layer core as
the mamba-rs pages state them (forward_mixed.rs 0.3.1, steps F4a-F4e;
trainer.rs 0.7.3, A = -exp(a_log), zero initial state).
"""

import numpy as np
import pytest
import scipy.signal

import oracle
from mamba_selective_scan_gb300.inputs import make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_case(batch, T, D, N=4, W=4, seed=0, act="f32"):
    """A small case with every parameter non-trivial (random a_log, conv_b, D)."""
    inp = make_inputs(batch, T, D, act=act, seed=seed, d_state=N, d_conv=W)
    rng = np.random.default_rng(1000 + seed)
    a = {k: np.array(v, dtype=np.float64) for k, v in inp.arrays.items()}
    a["a_log"] = rng.uniform(-1.0, 1.5, size=(D, N))
    a["conv_b"] = rng.uniform(-0.3, 0.3, size=D)
    a["D"] = rng.uniform(0.5, 1.5, size=D)
    return a


def _silu(v):
    return v / (1.0 + np.exp(-v))


# --------------------------------------------------------------------------
# Finite differences: every gradient of L = sum(gated * d_gated)
# --------------------------------------------------------------------------

_FD_TARGETS = {
    "x": "d_x", "delta_raw": "d_delta_raw", "z": "dz", "B": "dB", "C": "dC",
    "conv_w": "d_conv_w", "conv_b": "d_conv_b", "dt_bias": "d_dt_bias",
    "a_log": "d_a_log", "D": "dD",
}


def _fd_grad(a, name, eps=1e-6):
    base = a[name]
    g = np.zeros_like(base)
    flat = base.reshape(-1)
    gflat = g.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        h = eps * max(1.0, abs(old))
        flat[i] = old + h
        lp = oracle.loss(a)
        flat[i] = old - h
        lm = oracle.loss(a)
        flat[i] = old
        gflat[i] = (lp - lm) / (2 * h)
    return g


@pytest.mark.parametrize("shape", [(1, 1, 4, 4), (2, 3, 4, 4), (1, 8, 8, 1),
                                   (2, 8, 4, 4), (1, 17, 4, 16)])
def test_every_gradient_matches_central_differences(shape):
    batch, T, D, N = shape
    a = _rand_case(batch, T, D, N=N, seed=T + D)
    g = oracle.backward(a)
    for name, gname in _FD_TARGETS.items():
        fd = _fd_grad(a, name)
        an = g[gname]
        scale = max(np.abs(fd).max(), 1e-12)
        err = np.abs(an - fd).max() / scale
        assert err < 2e-6, f"{gname} vs FD: normalised error {err:.3e}"


def test_du_matches_finite_differences_through_u():
    """du is dL/du through the D skip and the recurrence (not through conv).

    Perturbing u directly is not an oracle input, so pin du through the chain
    rule on conv_b: dL/dconv_b[d] = sum_t du[t] * silu'(c[t]).  With all conv
    taps zero, c = conv_b, so silu'(c) is a constant per channel.
    """
    a = _rand_case(2, 6, 4, N=4, seed=7)
    a["conv_w"][:] = 0.0
    g = oracle.backward(a)
    cb = a["conv_b"]
    s = 1 / (1 + np.exp(-cb))
    dsilu = s + cb * s * (1 - s)
    want = g["du"].sum(axis=(0, 1)) * dsilu
    fd = _fd_grad(a, "conv_b")
    assert np.allclose(want, fd, rtol=1e-6, atol=1e-9)


# --------------------------------------------------------------------------
# Forward: closed form, library routines, brute force
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N", [16, 32, 64])
def test_closed_form_constant_inputs(N):
    """conv_w = [0,0,0,w3], conv_b = 0 and constant x, delta, B, C give
    h_k = delta*B*u*(1 - dA^(k+1)) / (1 - dA) per lane after k+1 updates."""
    T, D = 50, 3
    a = _rand_case(1, T, D, N=N, seed=3)
    a["conv_w"][:] = 0.0
    a["conv_w"][:, 3] = [0.7, -0.4, 1.1]
    a["conv_b"][:] = 0.0
    x0 = np.array([0.9, -1.3, 0.4])
    a["x"][:] = x0[None, None, :]
    dr0 = np.array([-0.2, 0.3, 0.0])
    a["delta_raw"][:] = dr0[None, None, :]
    Bv = np.linspace(-1, 1, N)
    Cv = np.cos(np.arange(N))
    a["B"][:] = Bv
    a["C"][:] = Cv
    out = oracle.forward(a)
    k = np.arange(T)[:, None]
    for d in range(D):
        c = a["conv_w"][d, 3] * x0[d]
        u = c / (1 + np.exp(-c))
        delta = np.log1p(np.exp(dr0[d] + a["dt_bias"][d]))
        A = -np.exp(a["a_log"][d])
        dA = np.exp(delta * A)
        h = delta * Bv * u * (1 - dA[None, :] ** (k + 1)) / (1 - dA[None, :])
        y = h @ Cv + a["D"][d] * u
        assert np.allclose(out["y"][0, :, d], y, rtol=1e-12, atol=1e-13)
        assert np.allclose(out["u"][0, :, d], u, rtol=1e-14)


def test_conv_matches_numpy_convolve():
    """u = silu(causal conv): the conv is numpy.convolve(x, reversed taps),
    full mode, first T outputs (zero left padding, w[W-1] on the current token)."""
    a = _rand_case(2, 11, 5, N=4, seed=5)
    out = oracle.forward(a)
    for b in range(2):
        for d in range(5):
            c = np.convolve(a["x"][b, :, d], a["conv_w"][d, ::-1])[:11] + a["conv_b"][d]
            assert np.allclose(out["u"][b, :, d], _silu(c), rtol=1e-13, atol=1e-15)


def test_short_sequences_shorter_than_the_conv():
    for T in (1, 2, 3):
        a = _rand_case(1, T, 4, N=4, seed=T)
        out = oracle.forward(a)
        for d in range(4):
            c = np.convolve(a["x"][0, :, d], a["conv_w"][d, ::-1])[:T] + a["conv_b"][d]
            assert np.allclose(out["u"][0, :, d], _silu(c), rtol=1e-13)


def test_delta_is_softplus_of_raw_plus_bias():
    a = _rand_case(1, 9, 4, N=4, seed=9)
    a["delta_raw"][0, :, 0] = [-40, -5, -1, 0, 1, 5, 20, 40, 700]
    out = oracle.forward(a)
    v = a["delta_raw"] + a["dt_bias"]
    want = np.logaddexp(0.0, v)  # library form of log(1 + e^v)
    assert np.allclose(out["delta"], want, rtol=1e-14, atol=0)


def test_constant_delta_scan_is_a_linear_filter():
    """With delta constant in time each lane is the first-order IIR filter
    h_t = dA h_{t-1} + x_t: scipy.signal.lfilter([1], [1, -dA], x)."""
    T, D, N = 40, 3, 16
    a = _rand_case(2, T, D, N=N, seed=11)
    a["delta_raw"][:] = np.array([0.1, -0.7, 0.5])[None, None, :]
    K = 7
    out = oracle.forward(a, ckpt_chunk=K)
    for b in range(2):
        for d in range(D):
            u = out["u"][b, :, d]
            delta = out["delta"][b, 0, d]
            A = -np.exp(a["a_log"][d])
            y = a["D"][d] * u
            for n in range(N):
                dA = np.exp(delta * A[n])
                h = scipy.signal.lfilter([1.0], [1.0, -dA], delta * a["B"][b, :, n] * u)
                y = y + a["C"][b, :, n] * h
                # checkpoint c holds the state before step c*K
                for c in range(out["ckpt"].shape[1]):
                    want = 0.0 if c == 0 else h[c * K - 1]
                    assert abs(out["ckpt"][b, c, n, d] - want) <= 1e-12 * (1 + abs(want))
            assert np.allclose(out["y"][b, :, d], y, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("N", [16, 32, 64])
def test_time_varying_scan_matches_unrolled_sum(N):
    """Brute force: h_t = sum_{s<=t} exp(A (S_t - S_s)) delta_s B_s u_s with
    S the running sum of delta, for time-varying delta, B, u."""
    T, D = 12, 2
    a = _rand_case(1, T, D, N=N, seed=13)
    out = oracle.forward(a)
    for d in range(D):
        u = out["u"][0, :, d]
        delta = out["delta"][0, :, d]
        S = np.cumsum(delta)
        A = -np.exp(a["a_log"][d])
        for t in range(T):
            h = np.zeros(N)
            for s in range(t + 1):
                h += np.exp(A * (S[t] - S[s])) * delta[s] * a["B"][0, s] * u[s]
            y = a["C"][0, t] @ h + a["D"][d] * u[t]
            assert abs(out["y"][0, t, d] - y) <= 1e-11 * (1 + abs(y))
            g = y * _silu(a["z"][0, t, d])
            assert abs(out["gated"][0, t, d] - g) <= 1e-11 * (1 + abs(g))


def test_memoryless_limit_when_A_is_very_negative():
    """a_log large -> dA = 0 -> h_t = delta_t B_t u_t -> y = delta u (C.B) + D u."""
    a = _rand_case(2, 10, 3, N=16, seed=17)
    a["a_log"][:] = 50.0
    out = oracle.forward(a)
    cb = np.einsum("btn,btn->bt", a["C"], a["B"])[:, :, None]
    want = out["delta"] * out["u"] * cb + a["D"] * out["u"]
    assert np.allclose(out["y"], want, rtol=1e-12, atol=1e-14)


def test_vanishing_step_leaves_only_the_skip():
    a = _rand_case(1, 10, 3, N=16, seed=19)
    a["delta_raw"][:] = -80.0
    out = oracle.forward(a)
    assert np.allclose(out["y"], a["D"] * out["u"], rtol=0, atol=1e-25)


def test_gate_becomes_identity_for_large_z():
    a = _rand_case(1, 10, 3, N=16, seed=21)
    a["z"][:] = 60.0
    out = oracle.forward(a)
    assert np.allclose(out["gated"], out["y"] * 60.0, rtol=1e-15)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

def test_scaling_B_and_inverse_scaling_C_leaves_y_unchanged():
    a = _rand_case(2, 15, 4, N=16, seed=23)
    y0 = oracle.forward(a)["y"]
    a2 = dict(a)
    a2["B"] = a["B"] * 3.0
    a2["C"] = a["C"] / 3.0
    assert np.allclose(oracle.forward(a2)["y"], y0, rtol=1e-12, atol=1e-13)
    a3 = dict(a)
    a3["C"] = a["C"] * -2.5
    o0 = oracle.forward(a)
    o3 = oracle.forward(a3)
    skip = a["D"] * o0["u"]
    assert np.allclose(o3["y"] - skip, -2.5 * (o0["y"] - skip), rtol=1e-12, atol=1e-13)


def test_gradients_are_linear_in_d_gated():
    a = _rand_case(2, 9, 4, N=16, seed=25)
    rng = np.random.default_rng(5)
    g1 = rng.standard_normal(a["x"].shape)
    g2 = rng.standard_normal(a["x"].shape)
    r1 = oracle.backward(a, d_gated=g1)
    r2 = oracle.backward(a, d_gated=g2)
    r = oracle.backward(a, d_gated=2.0 * g1 - 0.5 * g2)
    for k in oracle.GRAD_NAMES:
        want = 2.0 * r1[k] - 0.5 * r2[k]
        scale = max(np.abs(want).max(), 1e-300)
        assert np.abs(r[k] - want).max() / scale < 1e-12, k


# --------------------------------------------------------------------------
# Chunked recompute == sequential
# --------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 5, 64, 37])
def test_chunked_backward_equals_sequential(K):
    a = _rand_case(2, 37, 4, N=16, seed=27)
    seq = oracle.backward(a, chunk=0)
    ch = oracle.backward(a, chunk=K)
    for k in oracle.GRAD_NAMES:
        scale = max(np.abs(seq[k]).max(), 1e-300)
        assert np.abs(ch[k] - seq[k]).max() / scale < 1e-14, k


# --------------------------------------------------------------------------
# Channel masks (used by full-size sampled parity)
# --------------------------------------------------------------------------

def test_channel_mask_matches_zeroed_upstream_gradient():
    """Computing only masked channels equals the full oracle with d_gated
    zeroed outside the mask: per-channel outputs agree on the mask and dB, dC
    are the masked channels' contributions."""
    a = _rand_case(2, 20, 8, N=16, seed=29)
    mask = np.zeros(8, dtype=np.uint8)
    mask[[1, 6]] = 1
    gz = a["d_gated"] * mask[None, None, :]
    full = oracle.backward(a, d_gated=gz)
    part = oracle.backward(a, d_gated=gz, chan_mask=mask)
    on = mask.astype(bool)
    for k in ("d_x", "d_delta_raw", "dz", "du"):
        assert np.array_equal(part[k][:, :, on], full[k][:, :, on]), k
    for k in ("d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert np.array_equal(part[k][on], full[k][on]), k
    for k in ("dB", "dC"):
        assert np.allclose(part[k], full[k], rtol=1e-13, atol=1e-15), k
    fwd_full = oracle.forward(a)
    fwd_part = oracle.forward(a, chan_mask=mask)
    assert np.array_equal(fwd_part["gated"][:, :, on], fwd_full["gated"][:, :, on])


# --------------------------------------------------------------------------
# Independent cross-check: torch autograd in float64 on a per-step loop
# --------------------------------------------------------------------------

def test_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    a = _rand_case(2, 7, 4, N=16, seed=31)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for k, v in a.items() if k != "d_gated"}
    Bsz, T, D = a["x"].shape
    W = a["conv_w"].shape[1]
    xp = torch.nn.functional.pad(t["x"], (0, 0, W - 1, 0))
    c = t["conv_b"] + sum(t["conv_w"][:, k] * xp[:, k:k + T, :] for k in range(W))
    u = torch.nn.functional.silu(c)
    delta = torch.nn.functional.softplus(t["delta_raw"] + t["dt_bias"], threshold=1e9)
    A = -torch.exp(t["a_log"])  # [D, N]
    h = torch.zeros(Bsz, D, A.shape[1], dtype=torch.float64)
    ys = []
    for s in range(T):
        dA = torch.exp(delta[:, s, :, None] * A[None])
        h = dA * h + (delta[:, s, :] * u[:, s, :])[:, :, None] * t["B"][:, s, None, :]
        ys.append((h * t["C"][:, s, None, :]).sum(-1) + t["D"] * u[:, s, :])
    y = torch.stack(ys, 1)
    gated = y * torch.nn.functional.silu(t["z"])
    (gated * torch.tensor(a["d_gated"])).sum().backward()
    g = oracle.backward(a)
    pairs = {"d_x": "x", "d_delta_raw": "delta_raw", "dz": "z", "dB": "B", "dC": "C",
             "d_conv_w": "conv_w", "d_conv_b": "conv_b", "d_dt_bias": "dt_bias",
             "d_a_log": "a_log", "dD": "D"}
    for gname, iname in pairs.items():
        ref = t[iname].grad.numpy()
        assert np.allclose(g[gname], ref, rtol=1e-10, atol=1e-12), gname

"""Pins for the oracle's x_proj gradient path.

In the mamba-rs mixed-precision layer (forward_mixed.rs 0.3.1, the
per-layer loop: F4b x_proj of u into (dt_low, B, C), F4c dt_proj of dt_low
into delta_raw) u feeds both the selective scan and the x_proj GEMM, and the
backward adds the x_proj input gradient into d_u before the SiLU and conv1d
backward.  The layer core takes that extra gradient as ``d_u_extra``.

Pinned here: finite differences of the extended loss, and the chain rule
through a whole mini-layer (conv -> SiLU -> x_proj -> dt_proj -> scan ->
gate) differentiated by torch autograd in float64, against the two-phase
oracle computation (scan backward, then the x_proj GEMM's input gradient,
then the conv backward with it).
"""

import numpy as np
import pytest

import oracle
from mamba_selective_scan_gb300.inputs import make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _case(batch, T, D, N=4, seed=0):
    inp = make_inputs(batch, T, D, act="f32", seed=seed, d_state=N)
    rng = np.random.default_rng(3000 + seed)
    a = {k: np.array(v, dtype=np.float64) for k, v in inp.arrays.items()}
    a["a_log"] = rng.uniform(-1.0, 1.5, size=(D, N))
    a["conv_b"] = rng.uniform(-0.3, 0.3, size=D)
    a["D"] = rng.uniform(0.5, 1.5, size=D)
    gu = rng.standard_normal((batch, T, D))
    return a, gu


def _fd(a, gu, name, eps=1e-6):
    base = a[name]
    g = np.zeros_like(base)
    flat, gflat = base.reshape(-1), g.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        h = eps * max(1.0, abs(old))
        flat[i] = old + h
        lp = oracle.loss(a, d_u_extra=gu)
        flat[i] = old - h
        lm = oracle.loss(a, d_u_extra=gu)
        flat[i] = old
        gflat[i] = (lp - lm) / (2 * h)
    return g


@pytest.mark.parametrize("shape", [(1, 1, 4), (2, 5, 4), (1, 9, 8)])
def test_extra_u_gradient_matches_central_differences(shape):
    a, gu = _case(*shape, seed=sum(shape))
    g = oracle.backward(a, d_u_extra=gu)
    for name, gname in (("x", "d_x"), ("conv_w", "d_conv_w"), ("conv_b", "d_conv_b"),
                        ("delta_raw", "d_delta_raw"), ("B", "dB"), ("a_log", "d_a_log")):
        fd = _fd(a, gu, name)
        err = np.abs(g[gname] - fd).max() / max(np.abs(fd).max(), 1e-12)
        assert err < 2e-6, (gname, err)


def test_extra_u_gradient_touches_only_the_conv_side():
    a, gu = _case(2, 7, 4, seed=3)
    g0 = oracle.backward(a)
    g1 = oracle.backward(a, d_u_extra=gu)
    for k in ("d_delta_raw", "dz", "du", "dB", "dC", "d_dt_bias", "d_a_log", "dD"):
        assert np.array_equal(g0[k], g1[k]), k
    for k in ("d_x", "d_conv_w", "d_conv_b"):
        assert not np.allclose(g0[k], g1[k]), k


def test_two_phase_backward_through_x_proj_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    Bsz, T, D, N, R = 2, 6, 8, 4, 3
    a, _ = _case(Bsz, T, D, N=N, seed=11)
    rng = np.random.default_rng(12)
    Wx = rng.standard_normal((D, R + 2 * N)) * 0.3     # x_proj: u [.., D] -> [.., R + 2N]
    Wdt = rng.standard_normal((R, D)) * 0.3            # dt_proj: dt_low [.., R] -> [.., D]

    # torch: the whole mini-layer, B, C and delta_raw computed from u
    t = {k: torch.tensor(a[k], requires_grad=True)
         for k in ("x", "z", "conv_w", "conv_b", "dt_bias", "a_log", "D")}
    W = 4
    xp = torch.nn.functional.pad(t["x"], (0, 0, W - 1, 0))
    c = t["conv_b"] + sum(t["conv_w"][:, k] * xp[:, k:k + T, :] for k in range(W))
    u = torch.nn.functional.silu(c)
    xdbl = u @ torch.tensor(Wx)
    dt_low, Bm, Cm = xdbl[..., :R], xdbl[..., R:R + N], xdbl[..., R + N:]
    delta_raw = dt_low @ torch.tensor(Wdt)
    delta = torch.nn.functional.softplus(delta_raw + t["dt_bias"], threshold=1e9)
    A = -torch.exp(t["a_log"])
    h = torch.zeros(Bsz, D, N, dtype=torch.float64)
    ys = []
    for s in range(T):
        dA = torch.exp(delta[:, s, :, None] * A[None])
        h = dA * h + (delta[:, s, :] * u[:, s, :])[:, :, None] * Bm[:, s, None, :]
        ys.append((h * Cm[:, s, None, :]).sum(-1) + t["D"] * u[:, s, :])
    gated = torch.stack(ys, 1) * torch.nn.functional.silu(t["z"])
    (gated * torch.tensor(a["d_gated"])).sum().backward()

    # oracle, two phases: the scan's backward with B, C, delta_raw as inputs,
    # then the x_proj/dt_proj GEMMs' input gradient, then the conv side
    b = dict(a)
    b["B"] = xdbl[..., R:R + N].detach().numpy().copy()
    b["C"] = xdbl[..., R + N:].detach().numpy().copy()
    b["delta_raw"] = delta_raw.detach().numpy().copy()
    g1 = oracle.backward(b)
    d_dt_low = g1["d_delta_raw"] @ Wdt.T
    d_xdbl = np.concatenate([d_dt_low, g1["dB"], g1["dC"]], axis=-1)
    d_u_xproj = d_xdbl @ Wx.T
    g2 = oracle.backward(b, d_u_extra=d_u_xproj)
    for gname, leaf in (("d_x", "x"), ("dz", "z"), ("d_conv_w", "conv_w"),
                        ("d_conv_b", "conv_b"), ("d_dt_bias", "dt_bias"),
                        ("d_a_log", "a_log"), ("dD", "D")):
        assert np.allclose(g2[gname], t[leaf].grad.numpy(), rtol=1e-10, atol=1e-12), gname

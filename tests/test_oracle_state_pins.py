"""Pins for the oracle's carried state: the SSM state before the first step
and the conv inputs of the steps before it, the same two quantities at the
end of the window, and their gradients.

The mamba-rs pages carry both across calls: the per-layer conv1d of the
mixed-precision forward (forward_mixed.rs 0.3.1, step F4a) reads and
updates a conv state, the selective scan (step F4d) reads and writes the
SSM state, and the trainer (trainer.rs 0.7.3) keeps these between windows
and zeroes them on reset.  What fixes the semantics, independently of the
oracle's own code:

* finite differences of the extended loss, for every input including the
  carried state;
* window chaining: cutting a sequence in two and running the second window
  from the first one's state outputs must give exactly the one-window
  results, forward and backward;
* closed forms (a pure decay of the carried state when u = 0) and a library
  routine (numpy.convolve over the carried inputs followed by x);
* torch autograd in float64 on a per-step loop that starts from the state;
* the empty window, where the outputs are the inputs.
"""

import numpy as np
import pytest

import oracle
from mamba_selective_scan_gb300.inputs import make_inputs, make_state_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

STATE_KW = ("ssm_state", "conv_state", "d_ssm_state_out", "d_conv_state_out")


def _case(batch, T, D, N=4, W=4, seed=0):
    inp = make_inputs(batch, T, D, act="f32", seed=seed, d_state=N, d_conv=W)
    rng = np.random.default_rng(2000 + seed)
    a = {k: np.array(v, dtype=np.float64) for k, v in inp.arrays.items()}
    a["a_log"] = rng.uniform(-1.0, 1.5, size=(D, N))
    a["conv_b"] = rng.uniform(-0.3, 0.3, size=D)
    a["D"] = rng.uniform(0.5, 1.5, size=D)
    st = {k: np.array(v, dtype=np.float64)
          for k, v in make_state_inputs(batch, D, "f32", seed, N, W).items()}
    return a, st


def _slice_t(a, t0, t1):
    out = dict(a)
    for k in ("x", "delta_raw", "z", "B", "C", "d_gated"):
        out[k] = np.ascontiguousarray(a[k][:, t0:t1])
    return out


# --------------------------------------------------------------------------
# Finite differences of the extended loss
# --------------------------------------------------------------------------

def _fd(a, st, where, name, eps=1e-6):
    base = (a if where == "a" else st)[name]
    g = np.zeros_like(base)
    flat, gflat = base.reshape(-1), g.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        h = eps * max(1.0, abs(old))
        flat[i] = old + h
        lp = oracle.loss(a, **st)
        flat[i] = old - h
        lm = oracle.loss(a, **st)
        flat[i] = old
        gflat[i] = (lp - lm) / (2 * h)
    return g


_TARGETS = [("a", "x", "d_x"), ("a", "delta_raw", "d_delta_raw"), ("a", "z", "dz"),
            ("a", "B", "dB"), ("a", "C", "dC"), ("a", "conv_w", "d_conv_w"),
            ("a", "conv_b", "d_conv_b"), ("a", "dt_bias", "d_dt_bias"),
            ("a", "a_log", "d_a_log"), ("a", "D", "dD"),
            ("s", "ssm_state", "d_ssm_state"), ("s", "conv_state", "d_conv_state")]


@pytest.mark.parametrize("shape", [(1, 1, 4, 4), (2, 2, 4, 4), (1, 3, 4, 4),
                                   (2, 6, 4, 4), (1, 9, 4, 16)])
def test_every_gradient_with_carried_state_matches_central_differences(shape):
    batch, T, D, N = shape
    a, st = _case(batch, T, D, N=N, seed=3 * T + D)
    g = oracle.backward(a, **st)
    for where, name, gname in _TARGETS:
        fd = _fd(a, st, where, name)
        scale = max(np.abs(fd).max(), 1e-12)
        err = np.abs(g[gname] - fd).max() / scale
        assert err < 2e-6, f"{gname} vs FD: normalised error {err:.3e}"


def test_state_gradients_vanish_only_without_upstream_gradients():
    """The carried state reaches every later output, so d_ssm_state is
    nonzero with d_gated alone; with every upstream gradient zero, every
    gradient is zero."""
    a, st = _case(2, 5, 4, seed=4)
    g = oracle.backward(a, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    assert np.abs(g["d_ssm_state"]).max() > 0
    a0 = dict(a)
    a0["d_gated"] = np.zeros_like(a["d_gated"])
    g0 = oracle.backward(a0, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    for k in oracle.GRAD_NAMES + oracle.STATE_GRAD_NAMES:
        assert np.abs(g0[k]).max() == 0.0, k


# --------------------------------------------------------------------------
# Window chaining
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,T1", [(11, 5), (11, 1), (11, 2), (11, 3), (11, 0), (11, 11),
                                  (2, 1), (8, 4)])
def test_two_windows_equal_one_window(T, T1):
    a, st = _case(2, T, 4, N=4, seed=T + 7 * T1)
    full_f = oracle.forward(a, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    full_g = oracle.backward(a, **st)

    a1, a2 = _slice_t(a, 0, T1), _slice_t(a, T1, T)
    f1 = oracle.forward(a1, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    f2 = oracle.forward(a2, ssm_state=f1["ssm_state_out"], conv_state=f1["conv_state_out"])
    for k in ("gated", "y", "u", "delta"):
        got = np.concatenate([f1[k], f2[k]], axis=1)
        assert np.allclose(got, full_f[k], rtol=1e-12, atol=1e-12), k
    for k in ("ssm_state_out", "conv_state_out"):
        assert np.allclose(f2[k], full_f[k], rtol=1e-12, atol=1e-12), k

    # backward: the second window first; its state-input gradients are the
    # first window's upstream gradients on its state outputs
    g2 = oracle.backward(a2, ssm_state=f1["ssm_state_out"], conv_state=f1["conv_state_out"],
                         d_ssm_state_out=st["d_ssm_state_out"],
                         d_conv_state_out=st["d_conv_state_out"])
    g1 = oracle.backward(a1, ssm_state=st["ssm_state"], conv_state=st["conv_state"],
                         d_ssm_state_out=g2["d_ssm_state"], d_conv_state_out=g2["d_conv_state"])
    for k in ("d_x", "d_delta_raw", "dz", "du", "dB", "dC"):
        got = np.concatenate([g1[k], g2[k]], axis=1)
        assert np.allclose(got, full_g[k], rtol=1e-10, atol=1e-12), k
    for k in ("d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert np.allclose(g1[k] + g2[k], full_g[k], rtol=1e-10, atol=1e-12), k
    for k in oracle.STATE_GRAD_NAMES:
        assert np.allclose(g1[k], full_g[k], rtol=1e-10, atol=1e-12), k


def test_many_windows_of_one_step_equal_one_window():
    a, st = _case(1, 9, 4, N=16, seed=13)
    full = oracle.forward(a, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    h, c = st["ssm_state"], st["conv_state"]
    ys = []
    for t in range(9):
        f = oracle.forward(_slice_t(a, t, t + 1), ssm_state=h, conv_state=c)
        ys.append(f["gated"])
        h, c = f["ssm_state_out"], f["conv_state_out"]
    assert np.allclose(np.concatenate(ys, axis=1), full["gated"], rtol=1e-12, atol=1e-13)
    assert np.allclose(h, full["ssm_state_out"], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Closed forms and library routines
# --------------------------------------------------------------------------

def test_pure_decay_of_the_carried_state():
    """x = 0, conv_b = 0 and a zero conv state give u = 0, so each lane only
    decays: h_t[n] = exp(A[n] * sum_{s<=t} delta_s) h_{-1}[n] and
    y_t = sum_n C_t[n] h_t[n]."""
    a, st = _case(2, 12, 3, N=16, seed=21)
    a["x"][:] = 0.0
    a["conv_b"][:] = 0.0
    out = oracle.forward(a, ssm_state=st["ssm_state"], conv_state=np.zeros_like(st["conv_state"]))
    A = -np.exp(a["a_log"])                                      # [D, N]
    cums = np.cumsum(np.logaddexp(0.0, a["delta_raw"] + a["dt_bias"]), axis=1)  # [B,T,D]
    h = np.exp(cums[..., None] * A[None, None]) * np.transpose(st["ssm_state"], (0, 2, 1))[:, None]
    y = np.einsum("btdn,btn->btd", h, a["C"])
    assert np.allclose(out["y"], y, rtol=1e-12, atol=1e-13)
    assert np.allclose(out["ssm_state_out"], np.transpose(h[:, -1], (0, 2, 1)), rtol=1e-12)


def test_conv_over_carried_inputs_matches_numpy_convolve():
    """The conv runs over the carried inputs followed by x: numpy.convolve
    (full mode) of that sequence with the reversed taps, outputs W-1..W-2+T."""
    for T in (1, 2, 3, 10):
        a, st = _case(2, T, 5, N=4, seed=30 + T)
        out = oracle.forward(a, conv_state=st["conv_state"])
        for b in range(2):
            for d in range(5):
                seq = np.concatenate([st["conv_state"][b, :, d], a["x"][b, :, d]])
                c = np.convolve(seq, a["conv_w"][d, ::-1])[3:3 + T] + a["conv_b"][d]
                u = c / (1 + np.exp(-c))
                assert np.allclose(out["u"][b, :, d], u, rtol=1e-13, atol=1e-15)
                assert np.array_equal(out["conv_state_out"][b, :, d], seq[-3:])


def test_empty_window_passes_the_state_through():
    a, st = _case(2, 0, 4, N=4, seed=40)
    f = oracle.forward(a, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    assert np.array_equal(f["ssm_state_out"], st["ssm_state"])
    assert np.array_equal(f["conv_state_out"], st["conv_state"])
    g = oracle.backward(a, **st)
    assert np.array_equal(g["d_ssm_state"], st["d_ssm_state_out"])
    assert np.array_equal(g["d_conv_state"], st["d_conv_state_out"])
    for k in ("d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert np.abs(g[k]).max() == 0.0


# --------------------------------------------------------------------------
# Independent cross-check: torch autograd from a carried state
# --------------------------------------------------------------------------

def test_backward_with_state_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    a, st = _case(2, 6, 4, N=16, seed=50)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for k, v in a.items() if k != "d_gated"}
    h0 = torch.tensor(st["ssm_state"], requires_grad=True)          # [B, N, D]
    c0 = torch.tensor(st["conv_state"], requires_grad=True)         # [B, W-1, D]
    Bsz, T, D = a["x"].shape
    W = a["conv_w"].shape[1]
    xp = torch.cat([c0, t["x"]], dim=1)
    c = t["conv_b"] + sum(t["conv_w"][:, k] * xp[:, k:k + T, :] for k in range(W))
    u = torch.nn.functional.silu(c)
    delta = torch.nn.functional.softplus(t["delta_raw"] + t["dt_bias"], threshold=1e9)
    A = -torch.exp(t["a_log"])
    h = h0.transpose(1, 2)                                          # [B, D, N]
    ys = []
    for s in range(T):
        dA = torch.exp(delta[:, s, :, None] * A[None])
        h = dA * h + (delta[:, s, :] * u[:, s, :])[:, :, None] * t["B"][:, s, None, :]
        ys.append((h * t["C"][:, s, None, :]).sum(-1) + t["D"] * u[:, s, :])
    y = torch.stack(ys, 1)
    gated = y * torch.nn.functional.silu(t["z"])
    L = ((gated * torch.tensor(a["d_gated"])).sum()
         + (h.transpose(1, 2) * torch.tensor(st["d_ssm_state_out"])).sum()
         + (xp[:, -(W - 1):] * torch.tensor(st["d_conv_state_out"])).sum())
    L.backward()
    g = oracle.backward(a, **st)
    pairs = {"d_x": t["x"], "d_delta_raw": t["delta_raw"], "dz": t["z"], "dB": t["B"],
             "dC": t["C"], "d_conv_w": t["conv_w"], "d_conv_b": t["conv_b"],
             "d_dt_bias": t["dt_bias"], "d_a_log": t["a_log"], "dD": t["D"],
             "d_ssm_state": h0, "d_conv_state": c0}
    for gname, leaf in pairs.items():
        assert np.allclose(g[gname], leaf.grad.numpy(), rtol=1e-10, atol=1e-12), gname


@pytest.mark.parametrize("K", [1, 3, 4])
def test_chunked_backward_with_state_equals_sequential(K):
    a, st = _case(2, 10, 4, N=4, seed=60 + K)
    seq = oracle.backward(a, **st)
    chk = oracle.backward(a, chunk=K, **st)
    for k in oracle.GRAD_NAMES + oracle.STATE_GRAD_NAMES:
        assert np.allclose(chk[k], seq[k], rtol=1e-12, atol=1e-13), k


def test_checkpoint_zero_is_the_carried_state():
    a, st = _case(1, 10, 4, N=4, seed=70)
    f = oracle.forward(a, ckpt_chunk=4, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    assert np.array_equal(f["ckpt"][:, 0], st["ssm_state"])


@pytest.mark.parametrize("N", [32, 64])
def test_one_step_windows_chain_for_wider_states(N):
    """d_state 32 and 64 (the decode path): stepping one token at a time from
    the carried state equals one window, and the state after it is the
    brute-force sum h_{T-1} = exp(A S_{T-1}) h_{-1}
    + sum_s exp(A (S_{T-1} - S_s)) delta_s B_s u_s."""
    a, st = _case(1, 6, 3, N=N, seed=80 + N)
    full = oracle.forward(a, ssm_state=st["ssm_state"], conv_state=st["conv_state"])
    h, c = st["ssm_state"], st["conv_state"]
    ys = []
    for t in range(6):
        f = oracle.forward(_slice_t(a, t, t + 1), ssm_state=h, conv_state=c)
        ys.append(f["gated"])
        h, c = f["ssm_state_out"], f["conv_state_out"]
    assert np.allclose(np.concatenate(ys, axis=1), full["gated"], rtol=1e-12, atol=1e-13)
    for d in range(3):
        u, delta = full["u"][0, :, d], full["delta"][0, :, d]
        S = np.cumsum(delta)
        A = -np.exp(a["a_log"][d])
        want = np.exp(A * S[-1]) * st["ssm_state"][0, :, d]
        for s in range(6):
            want = want + np.exp(A * (S[-1] - S[s])) * delta[s] * a["B"][0, s] * u[s]
        assert np.allclose(full["ssm_state_out"][0, :, d], want, rtol=1e-11, atol=1e-12)
        assert np.allclose(h[0, :, d], want, rtol=1e-11, atol=1e-12)

"""Seeded synthetic inputs for the selective-scan layer core.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark. It draws random numbers and rounds them to the activation
dtype; it holds none of the layer core's arithmetic (no convolution, no
softplus of the forward, no scan).

Value recipe (the same for every workload unless a workload says otherwise):

* ``x`` (conv input), ``z`` (gate, pre-SiLU), ``d_gated`` ~ N(0, 1)
* ``conv_w`` ~ U(-0.5, 0.5), shape ``[d_inner, d_conv]``; ``conv_b`` = 0
* ``delta_raw`` ~ N(0, 0.5) (0.5 read as the standard deviation)
* ``dt_bias`` = softplus^-1(U[0.001, 0.1]), shape ``[d_inner]``
* ``a_log[d, n]`` = log(n + 1)  (so A = -(n + 1), the S4D-real initialisation)
* ``B``, ``C`` ~ N(0, 1), shape ``[batch, T, d_state]``; ``D`` = 1

Draw order from ``numpy.random.default_rng(seed)`` (PCG64) is fixed:
x, z, d_gated, conv_w, delta_raw, dt_bias, B, C.  Draws are float32;
activation tensors of a bf16 workload are then rounded to bf16 with
round-to-nearest-even, and both sides of every comparison see the rounded
values.  Parameters stay float32.

The long-sequence workload replaces the delta_raw draw: it draws
delta* ~ U[0.001, 0.01] in delta_raw's slot and sets
``delta_raw = softplus^-1(delta*) - dt_bias`` (then rounds to bf16), so that
the step size lands near [0.001, 0.01] and decay across chunk checkpoints is
slow.

``random_params=True`` replaces the three per-channel parameters that the
recipe fixes (a_log, conv_b, D) with draws that differ per channel, from a
stream of their own (``default_rng([seed, 2])``, so the other draws are
unchanged), in this order:

* ``a_log[d, n]`` ~ U(-4, 3): A = -exp(a_log) spans [-20.1, -0.018], so that
  exp(delta A) reaches both nearly 1 (slow decay) and nearly 0 (no memory);
* ``conv_b[d]`` ~ U(-0.5, 0.5);
* ``D[d]`` ~ U(-1.5, 1.5).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D_STATE = 16
D_CONV = 4


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seq_len: int
    d_inner: int
    act: str  # "f32" or "bf16"
    seed: int
    d_state: int = D_STATE
    d_conv: int = D_CONV
    slow_delta: bool = False
    note: str = ""

    @property
    def elems(self) -> int:
        return self.batch * self.seq_len * self.d_inner


# The five workloads: a tiny all-f32 parity case, the trainer usage shape
# (batch 8, seq_len 128, d_model 256 -> d_inner 512), a Mamba-130M-like layer,
# a long-sequence layer with slow decay, and a Mamba-2.8B-like layer.
WORKLOADS = {
    w.name: w
    for w in (
        Workload("pr1_f32_b1_t64_d32", 1, 64, 32, "f32", 0,
                 note="all-f32 parity case"),
        Workload("trainer_b8_t128_d512", 8, 128, 512, "bf16", 1,
                 note="trainer usage shape, d_model 256"),
        Workload("m130m_b8_t2048_d1536", 8, 2048, 1536, "bf16", 2,
                 note="Mamba-130M-like layer core"),
        Workload("longseq_b1_t65536_d2048", 1, 65536, 2048, "bf16", 3,
                 slow_delta=True, note="delta in [0.001, 0.01]"),
        Workload("m2p8b_b4_t4096_d5120", 4, 4096, 5120, "bf16", 4,
                 note="Mamba-2.8B-like layer core"),
    )
}
WORKLOAD_ORDER = list(WORKLOADS)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even).

    Returns float32 values that are exactly representable in bf16.  Inputs
    must be finite (the recipe never draws NaN or Inf).
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are exactly bf16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _softplus_inverse(y: np.ndarray) -> np.ndarray:
    # inverse of log(1 + e^x): x = log(e^y - 1), computed in float64
    y = np.asarray(y, dtype=np.float64)
    return np.log(np.expm1(y))


ACT_NAMES = ("x", "delta_raw", "z", "B", "C", "d_gated")
PARAM_NAMES = ("conv_w", "conv_b", "dt_bias", "a_log", "D")


@dataclass
class Inputs:
    """Host copies (float32, already rounded for bf16 workloads)."""

    batch: int
    seq_len: int
    d_inner: int
    d_state: int
    d_conv: int
    act: str
    arrays: dict = field(default_factory=dict)

    def __getitem__(self, k):
        return self.arrays[k]

    def f64(self, k):
        return np.ascontiguousarray(self.arrays[k], dtype=np.float64)


def make_inputs(batch, seq_len, d_inner, act="bf16", seed=0, d_state=D_STATE,
                d_conv=D_CONV, slow_delta=False, random_params=False) -> Inputs:
    """Draw one seeded input set following the recipe in the module doc."""
    if act not in ("f32", "bf16"):
        raise ValueError(f"act must be 'f32' or 'bf16', got {act!r}")
    rng = np.random.default_rng(seed)
    bt = (batch, seq_len, d_inner)
    x = rng.standard_normal(bt, dtype=np.float32)
    z = rng.standard_normal(bt, dtype=np.float32)
    d_gated = rng.standard_normal(bt, dtype=np.float32)
    conv_w = rng.uniform(-0.5, 0.5, size=(d_inner, d_conv)).astype(np.float32)
    if slow_delta:
        delta_target = rng.uniform(0.001, 0.01, size=bt)
    else:
        delta_raw = (0.5 * rng.standard_normal(bt, dtype=np.float32)).astype(np.float32)
    dt_bias = _softplus_inverse(rng.uniform(0.001, 0.1, size=d_inner)).astype(np.float32)
    if slow_delta:
        delta_raw = (_softplus_inverse(delta_target) - dt_bias.astype(np.float64)).astype(np.float32)
        del delta_target
    Bm = rng.standard_normal((batch, seq_len, d_state), dtype=np.float32)
    Cm = rng.standard_normal((batch, seq_len, d_state), dtype=np.float32)
    conv_b = np.zeros(d_inner, dtype=np.float32)
    a_log = np.log(np.arange(1, d_state + 1, dtype=np.float64))[None, :].repeat(d_inner, 0)
    a_log = np.ascontiguousarray(a_log, dtype=np.float32)
    Dp = np.ones(d_inner, dtype=np.float32)
    if random_params:
        a_log, conv_b, Dp = draw_random_params(d_inner, d_state, seed)

    acts = dict(x=x, delta_raw=delta_raw, z=z, B=Bm, C=Cm, d_gated=d_gated)
    if act == "bf16":
        acts = {k: round_to_bf16(v) for k, v in acts.items()}
    arrays = dict(acts)
    arrays.update(conv_w=conv_w, conv_b=conv_b, dt_bias=dt_bias, a_log=a_log, D=Dp)
    return Inputs(batch, seq_len, d_inner, d_state, d_conv, act, arrays)


def draw_random_params(d_inner, d_state=D_STATE, seed=0):
    """Per-channel a_log [d_inner, d_state], conv_b and D [d_inner] (float32)
    drawn as the module doc states for ``random_params=True``."""
    rng = np.random.default_rng([seed, 2])
    a_log = rng.uniform(-4.0, 3.0, size=(d_inner, d_state)).astype(np.float32)
    conv_b = rng.uniform(-0.5, 0.5, size=d_inner).astype(np.float32)
    Dp = rng.uniform(-1.5, 1.5, size=d_inner).astype(np.float32)
    return a_log, conv_b, Dp


STATE_NAMES = ("ssm_state", "conv_state", "d_ssm_state_out", "d_conv_state_out")


def make_state_inputs(batch, d_inner, act="bf16", seed=0, d_state=D_STATE,
                      d_conv=D_CONV) -> dict:
    """Seeded carried state for a window that continues an earlier one.

    ``ssm_state`` [batch, d_state, d_inner] (float32) and ``conv_state``
    [batch, d_conv - 1, d_inner] (activation dtype: it holds earlier conv
    inputs), plus the upstream gradients of the window's state outputs,
    ``d_ssm_state_out`` (float32) and ``d_conv_state_out`` (activation
    dtype), all ~ N(0, 1) and drawn in that order from a stream of its own
    (``default_rng([seed, 1])``), so the activation draws of ``make_inputs``
    with the same seed are unchanged.
    """
    rng = np.random.default_rng([seed, 1])
    h = rng.standard_normal((batch, d_state, d_inner), dtype=np.float32)
    c = rng.standard_normal((batch, d_conv - 1, d_inner), dtype=np.float32)
    gh = rng.standard_normal((batch, d_state, d_inner), dtype=np.float32)
    gc = rng.standard_normal((batch, d_conv - 1, d_inner), dtype=np.float32)
    if act == "bf16":
        c, gc = round_to_bf16(c), round_to_bf16(gc)
    return dict(ssm_state=h, conv_state=c, d_ssm_state_out=gh, d_conv_state_out=gc)


def make_workload_inputs(name: str, random_params=False) -> Inputs:
    w = WORKLOADS[name]
    return make_inputs(w.batch, w.seq_len, w.d_inner, w.act, w.seed,
                       w.d_state, w.d_conv, w.slow_delta, random_params)

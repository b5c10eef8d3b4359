"""The seeded input recipe (host only, no GPU): the per-channel parameter
draws that the random-parameter parity cases rely on."""

import numpy as np

from mamba_selective_scan_gb300.inputs import make_inputs


def test_random_parameters_differ_per_channel_and_span_both_decay_limits():
    inp = make_inputs(1, 4, 64, act="f32", seed=3, random_params=True)
    a = inp["a_log"]
    assert a.shape == (64, 16) and a.dtype == np.float32
    assert len({tuple(r) for r in a}) == a.shape[0]       # a row of its own per channel
    A = -np.exp(a.astype(np.float64))
    assert A.max() > -0.03 and A.min() < -15.0            # exp(delta A) near 1 and near 0
    assert np.abs(inp["conv_b"]).max() > 0.3
    assert np.abs(inp["D"] - 1.0).max() > 1.0
    assert len(set(inp["D"].tolist())) == 64


def test_random_parameters_leave_the_other_draws_unchanged():
    a = make_inputs(2, 16, 32, act="bf16", seed=5)
    b = make_inputs(2, 16, 32, act="bf16", seed=5, random_params=True)
    for k in ("x", "delta_raw", "z", "B", "C", "d_gated", "conv_w", "dt_bias"):
        assert np.array_equal(a[k], b[k]), k
    assert not np.array_equal(a["a_log"], b["a_log"])

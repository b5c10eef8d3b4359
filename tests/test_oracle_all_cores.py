"""The all-core timing driver of the oracle (the benchmark's all-core CPU
baseline) gives the single-threaded oracle's results: the same bits for
every per-channel output (each channel runs the same code on one thread),
and dB/dC equal up to the order of the sum over channel blocks."""

import numpy as np

import oracle
from mamba_selective_scan_gb300.inputs import make_inputs


def test_all_core_driver_matches_the_single_threaded_oracle():
    inp = make_inputs(2, 37, 24, act="bf16", seed=4, random_params=True)
    par, used = oracle.forward_backward_all_cores(inp, threads=5)
    assert used == 5
    f = oracle.forward(inp)
    b = oracle.backward(inp)
    assert np.array_equal(par["gated"], f["gated"])
    for k in ("d_x", "d_delta_raw", "dz", "d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert np.array_equal(par[k], b[k]), k
    for k in ("dB", "dC"):
        assert np.abs(par[k] - b[k]).max() <= 1e-12 * np.abs(b[k]).max(), k


def test_more_threads_than_channels_is_fine():
    inp = make_inputs(1, 9, 8, act="f32", seed=2)
    par, used = oracle.forward_backward_all_cores(inp, threads=32)
    assert used <= 8
    assert np.array_equal(par["gated"], oracle.forward(inp)["gated"])

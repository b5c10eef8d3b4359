"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded, dtype-rounded inputs, element by element.

Small cases span several channel groups, chunks, time segments and ragged
tails; the five workloads run at full size in the launch configuration the
benchmark uses, compared on sampled channels (every per-channel output and
parameter gradient), and for dB/dC with the upstream gradient zeroed outside
the sampled channels so that the oracle's sampled sums are the exact answer.
"""

import numpy as np
import pytest

from mamba_selective_scan_gb300 import binding
from mamba_selective_scan_gb300.inputs import (WORKLOADS, make_inputs,
                                               make_workload_inputs)
from parity_util import assert_close, compare, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_selective_scan_gb300 import build
    build.build()


def _case(batch, T, D, act, seed, chunk=0, segments=0, fwd_segments=None, slow=False, tpc=0):
    inp = make_inputs(batch, T, D, act=act, seed=seed, slow_delta=slow)
    dev = to_device(inp)
    gpu = run_gpu(dev, chunk=chunk, segments=segments, fwd_segments=fwd_segments, tpc=tpc)
    ref = run_oracle(inp)
    return inp, gpu, ref


SMALL = [
    # batch, T, D, act, chunk, segments
    (1, 64, 32, "f32", 0, 0),
    (2, 200, 136, "f32", 16, 1),
    (2, 200, 136, "f32", 16, 3),
    (2, 200, 136, "bf16", 16, 0),
    (2, 200, 136, "bf16", 5, 4),
    (1, 1, 8, "f32", 0, 0),
    (1, 2, 8, "bf16", 0, 0),
    (3, 3, 16, "f32", 1, 0),
    (1, 7, 64, "f32", 2, 3),
    # chunks longer than the backward's 8-step tile: tiles forward from the
    # checkpoint, sub-checkpoints in the workspace, ragged last chunk
    (2, 97, 72, "bf16", 24, 2),
    (2, 97, 72, "f32", 32, 2),
    (2, 97, 72, "bf16", 40, 1),
    (1, 300, 72, "f32", 64, 2),
    (1, 700, 40, "bf16", 128, 3),
    (1, 600, 24, "f32", 256, 2),
    (1, 130, 200, "f32", 7, 5),
    (4, 33, 520, "bf16", 16, 2),
    (1, 200, 64, "bf16", 4, 12),  # more segments than a cluster of the split backward takes
]


@pytest.mark.parametrize("batch,T,D,act,chunk,segments", SMALL)
@pytest.mark.parametrize("tpc", [1, 2])
def test_small_cases_match_oracle(batch, T, D, act, chunk, segments, tpc):
    """Both backward main kernels (one and two threads per channel)."""
    inp, gpu, ref = _case(batch, T, D, act, seed=batch * 1000 + T + D, chunk=chunk,
                          segments=segments, tpc=tpc)
    assert_close(compare(gpu, ref, act),
                 f"B={batch} T={T} D={D} {act} K={chunk} S={segments} tpc={tpc}")


def test_forward_checkpoints_match_oracle_states():
    inp = make_inputs(2, 100, 64, act="f32", seed=5)
    dev = to_device(inp)
    gpu = run_gpu(dev, chunk=8, segments=4)
    import oracle
    ref = oracle.forward(inp, ckpt_chunk=8)["ckpt"]
    err = np.abs(gpu["ckpt"] - ref).max() / np.abs(ref).max()
    assert err < 1e-4, err


def test_segment_count_does_not_change_results_beyond_rounding():
    inp = make_inputs(2, 256, 128, act="f32", seed=9)
    dev = to_device(inp)
    a = run_gpu(dev, chunk=16, segments=1)
    for s in (2, 5, 16):
        b = run_gpu(dev, chunk=16, segments=s)
        for k in ("gated", "d_x", "dB", "dC", "d_a_log", "dD", "d_delta_raw", "dz"):
            scale = np.abs(a[k]).max()
            assert np.abs(a[k] - b[k]).max() <= 2e-5 * scale, (s, k)


def test_param_grads_accumulate_when_asked():
    from mamba_selective_scan_gb300 import binding
    inp = make_inputs(2, 50, 64, act="f32", seed=11)
    dev = to_device(inp)
    gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"],
                                        dev["C"], dev["conv_w"], dev["conv_b"],
                                        dev["dt_bias"], dev["a_log"], dev["D"])
    args = (dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"],
            dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"], ckpt, dev["d_gated"])
    g1 = binding.m3scan_bwd(*args)
    g2 = binding.m3scan_bwd(*args, accumulate_param_grads=True,
                            out={k: g1[k].clone() for k in
                                 ("d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD")})
    for k in ("d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        # float-atomic sums: equal up to the order of the additions
        assert (g2[k] - 2 * g1[k]).abs().max() <= 1e-6 * (2 * g1[k]).abs().max(), k
    # dB and dC are overwritten, not accumulated
    assert torch.allclose(g2["dB"], g1["dB"], rtol=1e-5, atol=1e-6)


def test_nonfinite_inputs_propagate_without_hanging():
    inp = make_inputs(1, 40, 64, act="f32", seed=13)
    inp.arrays["x"][0, 10, 5] = np.nan
    dev = to_device(inp)
    gpu = run_gpu(dev, chunk=8, segments=2)
    assert np.isnan(gpu["gated"][0, 10:, 5]).all()
    assert np.isfinite(gpu["gated"][0, :, 6]).all()


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_full_size_sampled(name):
    """Full-size workload in the benchmark's launch configuration (library
    defaults).  Per-channel outputs and parameter grads on sampled channels;
    dB/dC with d_gated zeroed outside the sample."""
    w = WORKLOADS[name]
    inp = make_workload_inputs(name)
    dev = to_device(inp)
    D = w.d_inner
    if w.elems <= 600_000:
        gpu = run_gpu(dev)
        ref = run_oracle(inp)
        assert_close(compare(gpu, ref, w.act), name)
        return
    chans = sorted({0, 1, 31, 32, 63, 64, D // 2 + 3, D - 65, D - 1})
    mask = np.zeros(D, dtype=np.uint8)
    mask[chans] = 1
    on = mask.astype(bool)
    # 1) unmasked upstream gradient: per-channel outputs on the sample
    gpu = run_gpu(dev)
    ref = run_oracle(inp, chan_mask=mask)

    def sel(k, a):
        if k in ("dB", "dC"):
            return a
        if a.ndim == 3:
            return a[:, :, on]
        return a[on]
    rep = compare(gpu, ref, w.act, select=sel)
    rep.pop("dB", None)
    rep.pop("dC", None)
    assert_close(rep, name + " (sampled channels)")
    # 2) upstream gradient only on the sample: dB, dC are the sample's sums
    gm = inp.arrays["d_gated"] * mask[None, None, :]
    dgm = to_device(type(inp)(inp.batch, inp.seq_len, inp.d_inner, inp.d_state, inp.d_conv,
                              inp.act, {"d_gated": gm}))["d_gated"]
    gpu2 = run_gpu(dev, d_gated=dgm, want_debug=False)
    ref2 = oracle_masked_dbdc(inp, mask)
    assert_close(compare(gpu2, ref2, w.act, keys=("dB", "dC")), name + " (dB/dC)")
    off = ~on
    for k in ("d_x", "d_delta_raw", "dz"):
        assert np.all(gpu2[k][:, :, off] == 0.0), k


def oracle_masked_dbdc(inp, mask):
    import oracle
    return oracle.backward(inp, chan_mask=mask)


WIDE = [
    # batch, T, D, act, chunk, segments, d_state
    (2, 100, 64, "f32", 8, 3, 32),
    (2, 97, 48, "bf16", 16, 2, 64),
    (1, 40, 24, "f32", 2, 4, 64),
    (3, 33, 136, "bf16", 0, 0, 32),
    (1, 3, 8, "f32", 1, 0, 64),
]


@pytest.mark.parametrize("batch,T,D,act,chunk,segments,N", WIDE)
def test_wider_states_match_oracle(batch, T, D, act, chunk, segments, N):
    """d_state 32 and 64 (the split kernels, d_state / 8 threads per channel)."""
    inp = make_inputs(batch, T, D, act=act, seed=batch * 100 + T + N, d_state=N)
    dev = to_device(inp)
    gpu = run_gpu(dev, chunk=chunk, segments=segments)
    ref = run_oracle(inp)
    assert_close(compare(gpu, ref, act), f"B={batch} T={T} D={D} {act} K={chunk} S={segments} N={N}")


def test_device_status_stays_clear():
    """Every tile copy of the split backward lands: the library's device
    status word reads zero after runs that use those kernels."""
    binding.m3scan_device_status()  # clear whatever earlier tests left
    for act, chunk, seg in (("bf16", 8, 3), ("f32", 16, 0)):
        inp, gpu, ref = _case(2, 130, 136, act, seed=77, chunk=chunk, segments=seg, tpc=2)
        assert_close(compare(gpu, ref, act), f"status case {act} K={chunk}")
    assert binding.m3scan_device_status() == 0
    # the same through a workspace's status block
    inp = make_inputs(2, 130, 136, act="bf16", seed=78)
    dev = to_device(inp)
    dims = binding.make_dims(2, 130, 136, chunk=8, segments=3)
    ws = binding.Workspace(binding.m3scan_plan(dims, binding.M3_BF16).workspace_bytes, "cuda:0")
    gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                        dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                        dev["a_log"], dev["D"], chunk=8, segments=3, workspace=ws)
    binding.m3scan_bwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"],
                       dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"], ckpt,
                       dev["d_gated"], chunk=8, segments=3, workspace=ws)
    assert binding.m3scan_get_status(ws) == 0


def test_bounded_tile_wait_gives_up_and_reports():
    """A block whose tile copy never lands gives up after about a second;
    the failure reaches the workspace's status block (m3scan_get_status:
    M3_ERR_TIMEOUT, and reading clears it) and the device status word; and
    the context stays usable for a normal call afterwards."""
    import time
    binding.m3scan_device_status()
    ws = binding.Workspace(4096, "cuda:0")
    other = binding.Workspace(4096, "cuda:0")
    s = torch.cuda.current_stream()
    assert binding.m3scan_get_status(ws) == 0
    t0 = time.time()
    binding.m3scan_selftest_wait_timeout(s.cuda_stream, workspace=ws)
    assert binding.STATUS[binding.m3scan_get_status(ws)] == "M3_ERR_TIMEOUT"
    assert time.time() - t0 < 30
    assert binding.m3scan_get_status(ws) == 0      # cleared by the read
    assert binding.m3scan_get_status(other) == 0   # another workspace saw nothing
    assert binding.m3scan_device_status() != 0
    assert binding.m3scan_device_status() == 0
    inp, gpu, ref = _case(1, 40, 24, "f32", seed=5, chunk=8, segments=2, tpc=2)
    assert_close(compare(gpu, ref, "f32"), "after the timeout diagnostic")
    assert binding.m3scan_device_status() == 0


@pytest.mark.parametrize("tpc", [1, 2])
@pytest.mark.parametrize("batch,T,D,act,chunk,segments", [
    (2, 200, 136, "f32", 16, 3),
    (2, 97, 72, "bf16", 32, 2),
    (4, 33, 520, "bf16", 16, 2),
    (1, 130, 200, "f32", 7, 1),
    (2, 300, 72, "f32", 64, 2),
])
def test_deterministic_matches_oracle_and_repeats_bit_for_bit(batch, T, D, act, chunk,
                                                                  segments, tpc):
    """dB and dC as fixed-order sums of the channel blocks' shares: within
    tolerance of the oracle, and two calls give identical bits for every
    output."""
    inp = make_inputs(batch, T, D, act=act, seed=batch * 77 + T + D)
    dev = to_device(inp)
    a = run_gpu(dev, chunk=chunk, segments=segments, tpc=tpc, det=True)
    b = run_gpu(dev, chunk=chunk, segments=segments, tpc=tpc, det=True)
    ref = run_oracle(inp)
    assert_close(compare(a, ref, act), f"deterministic B={batch} T={T} D={D} {act} tpc={tpc}")
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("batch,T,D,act,chunk,segments,N", [
    (2, 200, 136, "f32", 8, 5, 16),   # ragged channel block (136 = 64 + 64 + 8)
    (3, 97, 72, "bf16", 4, 6, 16),    # ragged last chunk and segment
    (1, 64, 520, "bf16", 8, 8, 16),
    (2, 120, 40, "f32", 8, 3, 32),
    (1, 96, 24, "bf16", 8, 4, 64),
])
def test_split_backward_finishes_sums_in_kernel(batch, T, D, act, chunk, segments, N):
    """Over 2-8 segments the split main kernel runs the segments of a channel
    block as one cluster, which sums the parameter shares, adds them into the
    outputs and finishes d_x at the segment boundaries (no tail kernel):
    within tolerance of the oracle, and against the
    fixed-order path of the deterministic mode the same bits for every
    per-element output and equal up to f32 reassociation for the sums."""
    from parity_util import norm_err
    inp = make_inputs(batch, T, D, act=act, seed=batch * 31 + T + D + N, d_state=N)
    dev = to_device(inp)
    dims = binding.make_dims(batch, T, D, d_state=N, chunk=chunk, segments=segments,
                             threads_per_channel=2)
    pl = binding.m3scan_plan(dims, binding.M3_F32 if act == "f32" else binding.M3_BF16)
    assert pl.bwd_segments > 1 and pl.bwd_threads_per_channel == N // 8
    assert pl.bwd_launches == 2  # aggregate + main
    a = run_gpu(dev, chunk=chunk, segments=segments, tpc=2)
    b = run_gpu(dev, chunk=chunk, segments=segments, tpc=2, det=True)
    assert_close(compare(a, run_oracle(inp), act),
                 f"cluster sums B={batch} T={T} D={D} N={N} {act}")
    for k in ("gated", "d_x", "d_delta_raw", "dz", "du"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("dB", "dC", "d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD"):
        assert norm_err(a[k], b[k]) <= 1e-6, k


def test_split_backward_in_kernel_sums_accumulate_when_asked():
    inp = make_inputs(2, 120, 136, act="f32", seed=21)
    dev = to_device(inp)
    kw = dict(chunk=8, segments=5, threads_per_channel=2)
    gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"],
                                        dev["C"], dev["conv_w"], dev["conv_b"],
                                        dev["dt_bias"], dev["a_log"], dev["D"], **kw)
    args = (dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"], dev["conv_w"],
            dev["conv_b"], dev["dt_bias"], dev["a_log"], dev["D"], ckpt, dev["d_gated"])
    keys = ("d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD")
    g1 = binding.m3scan_bwd(*args, **kw)
    prior = {k: torch.full_like(g1[k], 0.25) for k in keys}
    g2 = binding.m3scan_bwd(*args, accumulate_param_grads=True,
                            out={k: v.clone() for k, v in prior.items()}, **kw)
    for k in keys:
        want = g1[k] + prior[k]
        assert (g2[k] - want).abs().max() <= 1e-6 * want.abs().max(), k


@pytest.mark.parametrize("segments,tpc,det", [(4, 2, False), (4, 2, True), (3, 1, False)])
def test_back_to_back_calls_sharing_checkpoints_and_workspace(segments, tpc, det):
    """Forward/backward pairs of two input sets queued back to back on one
    stream, sharing the checkpoint and workspace buffers (a kernel that
    started before the previous call finished would overwrite what that call
    still reads; inside a call the kernels overlap by programmatic dependent
    launch), give the same results as the same calls with a synchronisation
    after each (the same bits, but for float-atomic sums without
    deterministic mode)."""
    from parity_util import norm_err, to_np
    kw = dict(chunk=8, segments=segments, threads_per_channel=tpc)
    sets = [to_device(make_inputs(2, 96, 136, act="bf16", seed=40 + i)) for i in range(2)]
    dims = binding.make_dims(2, 96, 136, deterministic=det, **kw)
    pl = binding.m3scan_plan(dims, binding.M3_BF16)
    ws = binding.Workspace(pl.workspace_bytes, "cuda:0")
    ckpt = torch.empty((2, pl.n_chunks, 16, 136), dtype=torch.float32, device="cuda:0")

    def pair(dev, sync):
        gated, _, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                                         dev["conv_w"], dev["conv_b"], dev["dt_bias"],
                                         dev["a_log"], dev["D"], ckpt=ckpt, workspace=ws, **kw)
        if sync:
            torch.cuda.synchronize()
        g = binding.m3scan_bwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                               dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"],
                               dev["D"], ckpt, dev["d_gated"], workspace=ws, deterministic=det,
                               **kw)
        if sync:
            torch.cuda.synchronize()
        return gated, g

    want = [pair(dev, True) for dev in sets]
    want = [(gt.clone(), {k: v.clone() for k, v in g.items()}) for gt, g in want]
    for _ in range(3):
        got = [pair(dev, False) for dev in sets]
        torch.cuda.synchronize()
        for (gt, g), (wgt, wg) in zip(got, want):
            assert torch.equal(gt, wgt)
            for k in wg:
                if det or k in ("d_x", "d_delta_raw", "dz"):
                    assert torch.equal(g[k], wg[k]), k
                else:
                    assert norm_err(to_np(g[k]), to_np(wg[k])) <= 1e-6, k


@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_empty_sequence_gives_zero_parameter_grads(act, accumulate):
    # T = 0: L has no terms, so every parameter gradient is zero (or, when
    # accumulating, the caller's values stay as they were)
    dt = torch.float32 if act == "f32" else torch.bfloat16
    dev = torch.device("cuda")
    Bsz, T, D, N = 2, 0, 16, 16
    x = torch.zeros((Bsz, T, D), dtype=dt, device=dev)
    bc = torch.zeros((Bsz, T, N), dtype=dt, device=dev)
    conv_w = torch.zeros((D, 4), device=dev)
    p = [torch.zeros(D, device=dev) for _ in range(3)]
    a_log = torch.zeros((D, N), device=dev)
    gated, ckpt, _ = binding.m3scan_fwd(x, x, x, bc, bc, conv_w, p[0], p[1], a_log, p[2])
    assert gated.numel() == 0
    prior = 7.0 if accumulate else float("nan")
    out = {"d_conv_w": torch.full((D, 4), prior, device=dev),
           "d_conv_b": torch.full((D,), prior, device=dev),
           "d_dt_bias": torch.full((D,), prior, device=dev),
           "d_a_log": torch.full((D, N), prior, device=dev),
           "dD": torch.full((D,), prior, device=dev)}
    g = binding.m3scan_bwd(x, x, x, bc, bc, conv_w, p[0], p[1], a_log, p[2], ckpt, x, out=out,
                           accumulate_param_grads=accumulate)
    torch.cuda.synchronize()
    for k in out:
        want = torch.full_like(out[k], 7.0) if accumulate else torch.zeros_like(out[k])
        assert torch.equal(g[k], want), k
    assert g["dB"].numel() == 0 and g["d_x"].numel() == 0

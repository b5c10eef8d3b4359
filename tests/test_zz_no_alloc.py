"""The allocation-free backward, m3scan_bwd_noalloc.

Some callers cannot allocate device memory (a host application that gives
the library a fixed memory budget and forbids allocation in its execution
path, or a latency-critical caller that cannot accept cudaMalloc's implicit
synchronisation).  m3scan_bwd_noalloc serves them with a fixed scratch array
inside the library.  These tests call it through the C ABI and compare it
with m3scan_bwd (caller-provided workspace), on two calls in a row, since
the scratch array is shared by every call and keeps the previous call's
contents.  The file sorts last so a run that stops at the first failure has
already run every other test.
"""

import numpy as np
import pytest

from mamba_selective_scan_gb300 import binding, build
from mamba_selective_scan_gb300.inputs import make_inputs

GRADS = ("d_x", "d_delta_raw", "dz", "du", "dB", "dC", "d_conv_w", "d_conv_b", "d_dt_bias",
         "d_a_log", "dD")


def test_noalloc_rejects_shapes_beyond_its_scratch_before_any_launch():
    # 64 x 24 x 4096 floats of parameter partials alone exceed 16 MiB; every
    # pointer is a fake address, so the call must fail before touching a device
    build.build()
    lib = binding.load()
    dims = binding.make_dims(64, 64, 4096, chunk=16, segments=1)
    plan = binding.m3scan_plan(dims, binding.M3_BF16)
    assert plan.workspace_bytes > binding.NOALLOC_SCRATCH_BYTES
    A = 1 << 20
    st = binding.raw_bwd_noalloc(dims, binding.M3_BF16, *([A] * 12), A, A, A, None,
                                 *([A] * 7), None)
    assert binding.STATUS[st] == "M3_ERR_WORKSPACE"
    assert hasattr(lib, "m3scan_bwd_noalloc")


@pytest.mark.gpu
@pytest.mark.parametrize("act,tpc,det", [
    ("bf16", 0, False), ("f32", 0, False),
    # the fixed-order sums keep the channel blocks' dB/dC shares in the
    # scratch as well; the second call must not read the first call's
    ("bf16", 1, True), ("f32", 2, True),
    ("bf16", 1, False), ("bf16", 2, False),
])
def test_noalloc_backward_matches_workspace_backward_twice(act, tpc, det):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from parity_util import TOL, norm_err, to_device, to_np
    build.build()
    batch, T, D = 2, 200, 136
    # per-channel parameters, so a wrong channel's a_log, conv_b or D shows
    inp = make_inputs(batch, T, D, act=act, seed=77, random_params=True)
    dev = to_device(inp)
    kw = dict(chunk=16, segments=3, threads_per_channel=tpc)
    gated, ckpt, _ = binding.m3scan_fwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"],
                                        dev["C"], dev["conv_w"], dev["conv_b"],
                                        dev["dt_bias"], dev["a_log"], dev["D"], **kw)
    ref = binding.m3scan_bwd(dev["x"], dev["delta_raw"], dev["z"], dev["B"], dev["C"],
                             dev["conv_w"], dev["conv_b"], dev["dt_bias"], dev["a_log"],
                             dev["D"], ckpt, dev["d_gated"], want_du=True, deterministic=det,
                             **kw)
    torch.cuda.synchronize()
    ref = {k: to_np(v) for k, v in ref.items()}
    dims = binding.make_dims(batch, T, D, deterministic=det, **kw)
    code = binding.M3_BF16 if act == "bf16" else binding.M3_F32
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        f32_keys = ("dB", "dC", "d_conv_w", "d_conv_b", "d_dt_bias", "d_a_log", "dD")
        out = {}
        for k in GRADS:  # NaN-filled: every element must be written by the call
            dt = torch.float32 if k in f32_keys else dev["x"].dtype
            out[k] = torch.full(ref[k].shape, float("nan"), dtype=dt, device=dev["x"].device)
        st = binding.raw_bwd_noalloc(
            dims, code, dev["x"].data_ptr(), dev["delta_raw"].data_ptr(), dev["z"].data_ptr(),
            dev["B"].data_ptr(), dev["C"].data_ptr(), dev["conv_w"].data_ptr(),
            dev["conv_b"].data_ptr(), dev["dt_bias"].data_ptr(), dev["a_log"].data_ptr(),
            dev["D"].data_ptr(), ckpt.data_ptr(), dev["d_gated"].data_ptr(),
            out["d_x"].data_ptr(), out["d_delta_raw"].data_ptr(), out["dz"].data_ptr(),
            out["du"].data_ptr(), out["dB"].data_ptr(), out["dC"].data_ptr(),
            out["d_conv_w"].data_ptr(), out["d_conv_b"].data_ptr(), out["d_dt_bias"].data_ptr(),
            out["d_a_log"].data_ptr(), out["dD"].data_ptr(), stream)
        assert st == 0, binding.m3scan_status_string(st)
        torch.cuda.synchronize()
        for k in GRADS:
            got = to_np(out[k])
            assert np.isfinite(got).all(), (call, k)
            if det:  # fixed-order sums: the same bits as the workspace call
                assert np.array_equal(got, ref[k]), (call, k)
            err = norm_err(got, ref[k])
            assert err <= TOL[act][k], (call, k, err)

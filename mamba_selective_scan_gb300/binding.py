"""Thin Python binding of the m3scan C ABI (include/m3scan.h).

Argument marshalling only: every step of the layer core runs in the CUDA
library.  PyTorch supplies device memory and the stream; outputs that the
caller does not pass are allocated here with ``torch.empty``.  If the
library cannot be loaded the calls raise -- there is no other path.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

M3_F32 = 0
M3_BF16 = 1

STATUS = {
    0: "M3_OK",
    1: "M3_ERR_NULL",
    2: "M3_ERR_DIMS",
    3: "M3_ERR_UNSUPPORTED",
    4: "M3_ERR_ALIGN",
    5: "M3_ERR_WORKSPACE",
    6: "M3_ERR_CUDA",
    7: "M3_ERR_TIMEOUT",
}

# bytes at the start of every workspace that hold the library's status block
STATUS_BYTES = 256

# every symbol include/m3scan.h declares
EXPORTS = ("m3scan_plan", "m3scan_fwd", "m3scan_bwd", "m3scan_fwd_state", "m3scan_bwd_state",
           "m3scan_bwd_scan", "m3scan_conv_bwd", "m3scan_decode", "m3scan_bwd_noalloc", "m3scan_status_string", "m3scan_last_cuda_error",
           "m3scan_version", "m3scan_get_status", "m3scan_device_status",
           "m3scan_selftest_wait_timeout")

# size of the library's own scratch array used by m3scan_bwd_noalloc
NOALLOC_SCRATCH_BYTES = 16 << 20


class M3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib_handle().m3scan_status_string(status).decode() if _LIB else STATUS.get(status)
        if status == 6 and _LIB:
            msg += f" ({_LIB.m3scan_last_cuda_error().decode()})"
        super().__init__(f"{where}: {msg}")


class M3Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seq_len", ctypes.c_int64),
                ("d_inner", ctypes.c_int64), ("d_state", ctypes.c_int64),
                ("d_conv", ctypes.c_int64), ("chunk", ctypes.c_int64),
                ("segments", ctypes.c_int64),
                ("accumulate_param_grads", ctypes.c_int32),
                ("threads_per_channel", ctypes.c_int32),
                ("bc_stride", ctypes.c_int64), ("dbc_stride", ctypes.c_int64),
                ("deterministic", ctypes.c_int32), ("reserved0", ctypes.c_int32)]


class M3Plan(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int64), ("n_chunks", ctypes.c_int64),
                ("fwd_segments", ctypes.c_int64), ("bwd_segments", ctypes.c_int64),
                ("ckpt_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("fwd_launches", ctypes.c_int32), ("bwd_launches", ctypes.c_int32),
                ("fwd_threads_per_channel", ctypes.c_int32),
                ("bwd_threads_per_channel", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class M3FwdState(ctypes.Structure):
    """m3_fwd_state: carried state in and out of a forward window."""
    _fields_ = [("ssm_state", ctypes.c_void_p), ("conv_state", ctypes.c_void_p),
                ("ssm_state_out", ctypes.c_void_p), ("conv_state_out", ctypes.c_void_p)]


class M3BwdState(ctypes.Structure):
    """m3_bwd_state: the conv state the forward used, the upstream gradients of
    the state outputs and the gradients of the state inputs."""
    _fields_ = [("conv_state", ctypes.c_void_p), ("d_ssm_state_out", ctypes.c_void_p),
                ("d_conv_state_out", ctypes.c_void_p), ("d_ssm_state", ctypes.c_void_p),
                ("d_conv_state", ctypes.c_void_p)]


_LIB = None
_LOCK = threading.Lock()
_vp = ctypes.c_void_p
_fp = ctypes.c_void_p  # float* passed as an address


def library_path() -> str:
    return _build.LIB_PATH


def _lib_handle(build_if_missing: bool = True):
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.LIB_PATH
            if build_if_missing and not os.path.exists(path):
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libm3scan not built: {path} is missing")
            lib = ctypes.CDLL(path)
            lib.m3scan_plan.restype = ctypes.c_int
            lib.m3scan_plan.argtypes = [ctypes.POINTER(M3Dims), ctypes.c_int,
                                        ctypes.POINTER(M3Plan)]
            lib.m3scan_fwd.restype = ctypes.c_int
            lib.m3scan_fwd.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int] + [_vp] * 5
                                       + [_fp] * 5 + [_vp, _vp, _fp, _vp, ctypes.c_size_t, _vp])
            lib.m3scan_bwd.restype = ctypes.c_int
            lib.m3scan_bwd.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int] + [_vp] * 5
                                       + [_fp] * 5 + [_fp, _vp] + [_vp] * 4 + [_fp] * 2
                                       + [_fp] * 5 + [_vp, ctypes.c_size_t, _vp])
            lib.m3scan_fwd_state.restype = ctypes.c_int
            lib.m3scan_fwd_state.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int] + [_vp] * 5
                                             + [_fp] * 5 + [_vp, _vp, _fp]
                                             + [ctypes.POINTER(M3FwdState)]
                                             + [_vp, ctypes.c_size_t, _vp])
            lib.m3scan_bwd_state.restype = ctypes.c_int
            lib.m3scan_bwd_state.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int] + [_vp] * 5
                                             + [_fp] * 5 + [_fp, _vp] + [_vp] * 4 + [_fp] * 2
                                             + [_fp] * 5 + [ctypes.POINTER(M3BwdState)]
                                             + [_vp, ctypes.c_size_t, _vp])
            lib.m3scan_bwd_scan.restype = ctypes.c_int
            lib.m3scan_bwd_scan.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int] + [_vp] * 5
                                            + [_fp] * 5 + [_fp, _vp] + [_vp] * 3 + [_fp] * 5
                                            + [ctypes.POINTER(M3BwdState)]
                                            + [_vp, ctypes.c_size_t, _vp])
            lib.m3scan_conv_bwd.restype = ctypes.c_int
            lib.m3scan_conv_bwd.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int, _vp, _fp, _fp,
                                             _vp, _vp, _vp, _fp, _fp,
                                             ctypes.POINTER(M3BwdState),
                                             _vp, ctypes.c_size_t, _vp])
            lib.m3scan_decode.restype = ctypes.c_int
            lib.m3scan_decode.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int] + [_vp] * 5
                                          + [_fp] * 5 + [_fp, _vp, _vp, _vp, _vp])
            lib.m3scan_bwd_noalloc.restype = ctypes.c_int
            lib.m3scan_bwd_noalloc.argtypes = ([ctypes.POINTER(M3Dims), ctypes.c_int] + [_vp] * 5
                                               + [_fp] * 5 + [_fp, _vp] + [_vp] * 4
                                               + [_fp] * 2 + [_fp] * 5 + [_vp])
            lib.m3scan_status_string.restype = ctypes.c_char_p
            lib.m3scan_status_string.argtypes = [ctypes.c_int]
            lib.m3scan_last_cuda_error.restype = ctypes.c_char_p
            lib.m3scan_last_cuda_error.argtypes = []
            lib.m3scan_version.restype = ctypes.c_int32
            lib.m3scan_version.argtypes = []
            lib.m3scan_device_status.restype = ctypes.c_int
            lib.m3scan_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32)]
            lib.m3scan_get_status.restype = ctypes.c_int
            lib.m3scan_get_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int)]
            lib.m3scan_selftest_wait_timeout.restype = ctypes.c_int
            lib.m3scan_selftest_wait_timeout.argtypes = [_vp, _vp]
            _LIB = lib
    return _LIB


def load():
    """Load libm3scan (building it first if it is missing)."""
    return _lib_handle()


def make_dims(batch, seq_len, d_inner, d_state=16, d_conv=4, chunk=0, segments=0,
              accumulate_param_grads=False, bc_stride=0, dbc_stride=0,
              threads_per_channel=0, deterministic=False) -> M3Dims:
    return M3Dims(int(batch), int(seq_len), int(d_inner), int(d_state), int(d_conv),
                  int(chunk), int(segments), int(bool(accumulate_param_grads)),
                  int(threads_per_channel), int(bc_stride), int(dbc_stride),
                  int(bool(deterministic)), 0)


def m3scan_plan(dims: M3Dims, act: int) -> M3Plan:
    out = M3Plan()
    st = _lib_handle().m3scan_plan(ctypes.byref(dims), int(act), ctypes.byref(out))
    if st != 0:
        raise M3Error(st, "m3scan_plan")
    return out


def m3scan_status_string(status: int) -> str:
    return _lib_handle().m3scan_status_string(int(status)).decode()


def m3scan_version() -> int:
    return int(_lib_handle().m3scan_version())


def m3scan_selftest_wait_timeout(stream: int = 0, workspace=None) -> None:
    """Enqueue the diagnostic block whose tile wait never completes (it
    reports to the device word and, if given, to ``workspace``'s status
    block)."""
    ws = None if workspace is None else workspace.ptr
    st = _lib_handle().m3scan_selftest_wait_timeout(ws, ctypes.c_void_p(stream))
    if st != 0:
        raise M3Error(st, "m3scan_selftest_wait_timeout")


def m3scan_get_status(workspace, stream=None) -> int:
    """Status of the calls made with ``workspace`` (a ``Workspace``) since the
    last query, then cleared: 0 (M3_OK) or 7 (M3_ERR_TIMEOUT).  Waits for
    ``stream`` (default: the current torch stream)."""
    out = ctypes.c_int(0)
    st = _lib_handle().m3scan_get_status(workspace.ptr, _stream_handle(stream), ctypes.byref(out))
    if st != 0:
        raise M3Error(st, "m3scan_get_status")
    return int(out.value)


def m3scan_device_status() -> int:
    """Device status since the last query (0 = every kernel ran normally),
    then cleared; waits for the device's queued work."""
    out = ctypes.c_int32(0)
    st = _lib_handle().m3scan_device_status(ctypes.byref(out))
    if st != 0:
        raise M3Error(st, "m3scan_device_status")
    return int(out.value)


def raw_fwd(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D,
            gated, y_dbg, ckpt, workspace, workspace_bytes, stream) -> int:
    """Call m3scan_fwd with integer addresses; returns the status code."""
    return _lib_handle().m3scan_fwd(ctypes.byref(dims), int(act), x, delta_raw, z, Bm, Cm,
                                    conv_w, conv_b, dt_bias, a_log, D, gated, y_dbg, ckpt,
                                    workspace, int(workspace_bytes), stream)


def raw_bwd(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
            d_gated, d_x, d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b, d_dt_bias,
            d_a_log, dD, workspace, workspace_bytes, stream) -> int:
    """Call m3scan_bwd with integer addresses; returns the status code."""
    return _lib_handle().m3scan_bwd(ctypes.byref(dims), int(act), x, delta_raw, z, Bm, Cm,
                                    conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated, d_x,
                                    d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b,
                                    d_dt_bias, d_a_log, dD, workspace, int(workspace_bytes),
                                    stream)


def raw_fwd_state(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D,
                  gated, y_dbg, ckpt, state, workspace, workspace_bytes, stream) -> int:
    """Call m3scan_fwd_state (``state`` an M3FwdState or None); returns the
    status code."""
    sp = ctypes.byref(state) if state is not None else None
    return _lib_handle().m3scan_fwd_state(ctypes.byref(dims), int(act), x, delta_raw, z, Bm, Cm,
                                          conv_w, conv_b, dt_bias, a_log, D, gated, y_dbg, ckpt,
                                          sp, workspace, int(workspace_bytes), stream)


def raw_bwd_state(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                  d_gated, d_x, d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b, d_dt_bias,
                  d_a_log, dD, state, workspace, workspace_bytes, stream) -> int:
    """Call m3scan_bwd_state (``state`` an M3BwdState or None); returns the
    status code."""
    sp = ctypes.byref(state) if state is not None else None
    return _lib_handle().m3scan_bwd_state(ctypes.byref(dims), int(act), x, delta_raw, z, Bm, Cm,
                                          conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated, d_x,
                                          d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b,
                                          d_dt_bias, d_a_log, dD, sp, workspace,
                                          int(workspace_bytes), stream)


def raw_bwd_scan(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                 d_gated, du, d_delta_raw, dz, dB, dC, d_dt_bias, d_a_log, dD, state, workspace,
                 workspace_bytes, stream) -> int:
    """Call m3scan_bwd_scan (``state`` an M3BwdState or None); returns the
    status code."""
    sp = ctypes.byref(state) if state is not None else None
    return _lib_handle().m3scan_bwd_scan(ctypes.byref(dims), int(act), x, delta_raw, z, Bm, Cm,
                                         conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated, du,
                                         d_delta_raw, dz, dB, dC, d_dt_bias, d_a_log, dD, sp,
                                         workspace, int(workspace_bytes), stream)


def raw_conv_bwd(dims, act, x, conv_w, conv_b, du, du_extra, d_x, d_conv_w, d_conv_b, state,
                 workspace, workspace_bytes, stream) -> int:
    """Call m3scan_conv_bwd (``state`` an M3BwdState or None); returns the
    status code."""
    sp = ctypes.byref(state) if state is not None else None
    return _lib_handle().m3scan_conv_bwd(ctypes.byref(dims), int(act), x, conv_w, conv_b, du,
                                         du_extra, d_x, d_conv_w, d_conv_b, sp, workspace,
                                         int(workspace_bytes), stream)


def raw_decode(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D,
               ssm_state, conv_state, gated, y_dbg, stream) -> int:
    """Call m3scan_decode with integer addresses; returns the status code."""
    return _lib_handle().m3scan_decode(ctypes.byref(dims), int(act), x, delta_raw, z, Bm, Cm,
                                       conv_w, conv_b, dt_bias, a_log, D, ssm_state, conv_state,
                                       gated, y_dbg, stream)


def raw_bwd_noalloc(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D,
                    ckpt, d_gated, d_x, d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b,
                    d_dt_bias, d_a_log, dD, stream) -> int:
    """Call m3scan_bwd_noalloc (no workspace; the library's fixed scratch
    array is used) with integer addresses; returns the status code.  For
    callers that cannot allocate device memory themselves."""
    return _lib_handle().m3scan_bwd_noalloc(ctypes.byref(dims), int(act), x, delta_raw, z, Bm,
                                            Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                                            d_gated, d_x, d_delta_raw, dz, du_dbg, dB, dC,
                                            d_conv_w, d_conv_b, d_dt_bias, d_a_log, dD, stream)


# ---------------------------------------------------------------------------
# torch-tensor wrappers (allocation and pointer marshalling only)
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _act_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return M3_BF16
    if t.dtype == torch.float32:
        return M3_F32
    raise TypeError(f"activation dtype must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t, name, dtype=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Workspace:
    """A device workspace sized for a plan (reusable across calls).  Its
    status block (the first STATUS_BYTES) starts at zero, as the library
    requires."""

    def __init__(self, nbytes: int, device):
        torch = _torch()
        self.nbytes = max(int(nbytes), STATUS_BYTES)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.buf[:STATUS_BYTES].zero_()

    @property
    def ptr(self):
        return self.buf.data_ptr()


def plan_for(x, chunk=0, segments=0):
    Bsz, T, D = x.shape
    dims = make_dims(Bsz, T, D, chunk=chunk, segments=segments)
    return dims, m3scan_plan(dims, _act_code(x))


def m3scan_fwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, *, chunk=0,
               segments=0, gated=None, y_dbg=None, want_y=False, ckpt=None, workspace=None,
               stream=None, threads_per_channel=0):
    """Forward of the layer core.  Returns (gated, ckpt, y_dbg or None)."""
    return _fwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, chunk, segments,
                gated, y_dbg, want_y, ckpt, workspace, stream, None, threads_per_channel)[:3]


def m3scan_fwd_state(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, *,
                     ssm_state=None, conv_state=None, chunk=0, segments=0, gated=None,
                     y_dbg=None, want_y=False, ckpt=None, ssm_state_out=None,
                     conv_state_out=None, workspace=None, stream=None, threads_per_channel=0):
    """Forward of one window from a carried state (None = zero).  Returns
    (gated, ckpt, y_dbg or None, ssm_state_out [B,16,D] f32,
    conv_state_out [B,3,D] activation dtype)."""
    torch = _torch()
    Bsz, _, Dn = x.shape
    N, W = Bm.shape[-1], conv_w.shape[-1]
    if ssm_state_out is None:
        ssm_state_out = torch.empty((Bsz, N, Dn), dtype=torch.float32, device=x.device)
    if conv_state_out is None:
        conv_state_out = torch.empty((Bsz, W - 1, Dn), dtype=x.dtype, device=x.device)
    _check(ssm_state, "ssm_state", torch.float32, x.device)
    _check(conv_state, "conv_state", x.dtype, x.device)
    _check(ssm_state_out, "ssm_state_out", torch.float32, x.device)
    _check(conv_state_out, "conv_state_out", x.dtype, x.device)
    st = M3FwdState(_ptr(ssm_state), _ptr(conv_state), _ptr(ssm_state_out),
                    _ptr(conv_state_out))
    gated, ckpt, y_dbg = _fwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, chunk,
                              segments, gated, y_dbg, want_y, ckpt, workspace, stream, st,
                              threads_per_channel)[:3]
    return gated, ckpt, y_dbg, ssm_state_out, conv_state_out


def _fwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, chunk, segments, gated,
         y_dbg, want_y, ckpt, workspace, stream, state, tpc=0):
    torch = _torch()
    act = x.dtype
    dev = x.device
    for n, t in (("x", x), ("delta_raw", delta_raw), ("z", z), ("B", Bm), ("C", Cm)):
        _check(t, n, act, dev)
    for n, t in (("conv_w", conv_w), ("conv_b", conv_b), ("dt_bias", dt_bias),
                 ("a_log", a_log), ("D", D)):
        _check(t, n, torch.float32, dev)
    Bsz, T, Dn = x.shape
    dims = make_dims(Bsz, T, Dn, d_state=Bm.shape[-1], d_conv=conv_w.shape[-1], chunk=chunk,
                     segments=segments, threads_per_channel=tpc)
    code = _act_code(x)
    pl = m3scan_plan(dims, code)
    if gated is None:
        gated = torch.empty_like(x)
    if want_y and y_dbg is None:
        y_dbg = torch.empty_like(x)
    if ckpt is None:
        ckpt = torch.empty((Bsz, pl.n_chunks, Bm.shape[-1], Dn), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = Workspace(pl.workspace_bytes, dev)
    args = (dims, code, _ptr(x), _ptr(delta_raw), _ptr(z), _ptr(Bm), _ptr(Cm),
            _ptr(conv_w), _ptr(conv_b), _ptr(dt_bias), _ptr(a_log), _ptr(D),
            _ptr(gated), _ptr(y_dbg), _ptr(ckpt))
    tail = (workspace.ptr, workspace.nbytes, _stream_handle(stream))
    if state is None:
        st = raw_fwd(*args, *tail)
    else:
        st = raw_fwd_state(*args, state, *tail)
    if st != 0:
        raise M3Error(st, "m3scan_fwd" if state is None else "m3scan_fwd_state")
    return gated, ckpt, y_dbg


def m3scan_bwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated, *,
               chunk=0, segments=0, want_du=False, accumulate_param_grads=False, out=None,
               workspace=None, stream=None, threads_per_channel=0, deterministic=False):
    """Backward of the layer core.  Returns a dict of gradients (tensors).
    ``deterministic``: dB, dC and the parameter gradients as fixed-order sums
    (identical bits on every call, a larger workspace) instead of float-atomic
    sums; the per-element gradients are the same bits either way."""
    return _bwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated,
                chunk, segments, want_du, accumulate_param_grads, out, workspace, stream, None,
                threads_per_channel, deterministic)


def m3scan_bwd_state(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated,
                     *, conv_state=None, d_ssm_state_out=None, d_conv_state_out=None, chunk=0,
                     segments=0, want_du=False, accumulate_param_grads=False, out=None,
                     workspace=None, stream=None, threads_per_channel=0, deterministic=False):
    """Backward of one window made by ``m3scan_fwd_state``.  Returns the
    gradients of ``m3scan_bwd`` plus ``d_ssm_state`` [B,16,D] f32 and
    ``d_conv_state`` [B,3,D] (activation dtype)."""
    torch = _torch()
    Bsz, _, Dn = x.shape
    N, W = Bm.shape[-1], conv_w.shape[-1]
    o = dict(out or {})
    o.setdefault("d_ssm_state", torch.empty((Bsz, N, Dn), dtype=torch.float32, device=x.device))
    o.setdefault("d_conv_state", torch.empty((Bsz, W - 1, Dn), dtype=x.dtype, device=x.device))
    _check(conv_state, "conv_state", x.dtype, x.device)
    _check(d_ssm_state_out, "d_ssm_state_out", torch.float32, x.device)
    _check(d_conv_state_out, "d_conv_state_out", x.dtype, x.device)
    _check(o["d_ssm_state"], "d_ssm_state", torch.float32, x.device)
    _check(o["d_conv_state"], "d_conv_state", x.dtype, x.device)
    st = M3BwdState(_ptr(conv_state), _ptr(d_ssm_state_out), _ptr(d_conv_state_out),
                    _ptr(o["d_ssm_state"]), _ptr(o["d_conv_state"]))
    return _bwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated,
                chunk, segments, want_du, accumulate_param_grads, o, workspace, stream, st,
                threads_per_channel, deterministic)


def _bwd(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt, d_gated, chunk,
         segments, want_du, accumulate_param_grads, out, workspace, stream, state, tpc=0,
         det=False):
    torch = _torch()
    act = x.dtype
    dev = x.device
    for n, t in (("x", x), ("delta_raw", delta_raw), ("z", z), ("B", Bm), ("C", Cm),
                 ("d_gated", d_gated)):
        _check(t, n, act, dev)
    for n, t in (("conv_w", conv_w), ("conv_b", conv_b), ("dt_bias", dt_bias),
                 ("a_log", a_log), ("D", D), ("ckpt", ckpt)):
        _check(t, n, torch.float32, dev)
    Bsz, T, Dn = x.shape
    N = Bm.shape[-1]
    W = conv_w.shape[-1]
    dims = make_dims(Bsz, T, Dn, d_state=N, d_conv=W, chunk=chunk, segments=segments,
                     accumulate_param_grads=accumulate_param_grads, threads_per_channel=tpc,
                     deterministic=det)
    code = _act_code(x)
    pl = m3scan_plan(dims, code)
    o = dict(out or {})
    o.setdefault("d_x", torch.empty_like(x))
    o.setdefault("d_delta_raw", torch.empty_like(x))
    o.setdefault("dz", torch.empty_like(x))
    if want_du:
        o.setdefault("du", torch.empty_like(x))
    f32 = dict(dtype=torch.float32, device=dev)
    o.setdefault("dB", torch.empty((Bsz, T, N), **f32))
    o.setdefault("dC", torch.empty((Bsz, T, N), **f32))
    o.setdefault("d_conv_w", torch.zeros((Dn, W), **f32))
    o.setdefault("d_conv_b", torch.zeros((Dn,), **f32))
    o.setdefault("d_dt_bias", torch.zeros((Dn,), **f32))
    o.setdefault("d_a_log", torch.zeros((Dn, N), **f32))
    o.setdefault("dD", torch.zeros((Dn,), **f32))
    for k, v in o.items():
        _check(v, k, None, dev)
    if workspace is None:
        workspace = Workspace(pl.workspace_bytes, dev)
    args = (dims, code, _ptr(x), _ptr(delta_raw), _ptr(z), _ptr(Bm), _ptr(Cm),
            _ptr(conv_w), _ptr(conv_b), _ptr(dt_bias), _ptr(a_log), _ptr(D), _ptr(ckpt),
            _ptr(d_gated), _ptr(o["d_x"]), _ptr(o["d_delta_raw"]), _ptr(o["dz"]),
            _ptr(o.get("du")), _ptr(o["dB"]), _ptr(o["dC"]), _ptr(o["d_conv_w"]),
            _ptr(o["d_conv_b"]), _ptr(o["d_dt_bias"]), _ptr(o["d_a_log"]), _ptr(o["dD"]))
    tail = (workspace.ptr, workspace.nbytes, _stream_handle(stream))
    if state is None:
        st = raw_bwd(*args, *tail)
    else:
        st = raw_bwd_state(*args, state, *tail)
    if st != 0:
        raise M3Error(st, "m3scan_bwd" if state is None else "m3scan_bwd_state")
    return o


def m3scan_decode(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ssm_state,
                  conv_state, *, gated=None, y_dbg=None, want_y=False, stream=None):
    """Forward of a short window (x [B, T, D], typically T = 1) from the
    carried state, updating ``ssm_state`` [B, N, D] (f32) and ``conv_state``
    [B, 3, D] (activation dtype) in place.  Returns (gated, y_dbg or None)."""
    torch = _torch()
    act = x.dtype
    dev = x.device
    for n, t in (("x", x), ("delta_raw", delta_raw), ("z", z), ("B", Bm), ("C", Cm),
                 ("conv_state", conv_state)):
        _check(t, n, act, dev)
    for n, t in (("conv_w", conv_w), ("conv_b", conv_b), ("dt_bias", dt_bias),
                 ("a_log", a_log), ("D", D), ("ssm_state", ssm_state)):
        _check(t, n, torch.float32, dev)
    Bsz, T, Dn = x.shape
    dims = make_dims(Bsz, T, Dn, d_state=Bm.shape[-1], d_conv=conv_w.shape[-1])
    if gated is None:
        gated = torch.empty_like(x)
    if want_y and y_dbg is None:
        y_dbg = torch.empty_like(x)
    st = raw_decode(dims, _act_code(x), _ptr(x), _ptr(delta_raw), _ptr(z), _ptr(Bm), _ptr(Cm),
                    _ptr(conv_w), _ptr(conv_b), _ptr(dt_bias), _ptr(a_log), _ptr(D),
                    _ptr(ssm_state), _ptr(conv_state), _ptr(gated), _ptr(y_dbg),
                    _stream_handle(stream))
    if st != 0:
        raise M3Error(st, "m3scan_decode")
    return gated, y_dbg


def m3scan_bwd_two_phase(x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                         d_gated, du_extra_fn=None, *, conv_state=None, d_ssm_state_out=None,
                         d_conv_state_out=None, chunk=0, segments=0, bc_stride=0, dbc_stride=0,
                         dB=None, dC=None, accumulate_param_grads=False, stream=None,
                         threads_per_channel=0, deterministic=False):
    """The two-phase backward: m3scan_bwd_scan, then ``du_extra_fn(grads)``
    (the caller's x_proj/dt_proj GEMMs, given the scan's gradients; may
    return None), then m3scan_conv_bwd.  ``Bm``/``Cm`` may be column views
    of one x_proj output (``bc_stride`` its row length), ``dB``/``dC``
    column views of its gradient (``dbc_stride``).  Returns the gradient
    dict (with ``du`` and, when states are involved, ``d_ssm_state`` and
    ``d_conv_state``)."""
    torch = _torch()
    act = x.dtype
    dev = x.device
    Bsz, T, Dn = x.shape
    N, W = Bm.shape[-1], conv_w.shape[-1]
    dims = make_dims(Bsz, T, Dn, d_state=N, d_conv=W, chunk=chunk, segments=segments,
                     accumulate_param_grads=accumulate_param_grads, bc_stride=bc_stride,
                     dbc_stride=dbc_stride, threads_per_channel=threads_per_channel,
                     deterministic=deterministic)
    code = _act_code(x)
    pl = m3scan_plan(dims, code)
    ws = Workspace(pl.workspace_bytes, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    o = {"du": torch.empty_like(x), "d_delta_raw": torch.empty_like(x), "dz": torch.empty_like(x),
         "dB": dB if dB is not None else torch.empty((Bsz, T, N), **f32),
         "dC": dC if dC is not None else torch.empty((Bsz, T, N), **f32),
         "d_dt_bias": torch.zeros((Dn,), **f32), "d_a_log": torch.zeros((Dn, N), **f32),
         "dD": torch.zeros((Dn,), **f32), "d_x": torch.empty_like(x),
         "d_conv_w": torch.zeros((Dn, W), **f32), "d_conv_b": torch.zeros((Dn,), **f32),
         "d_ssm_state": torch.empty((Bsz, N, Dn), **f32),
         "d_conv_state": torch.empty((Bsz, W - 1, Dn), dtype=act, device=dev)}
    st = M3BwdState(_ptr(conv_state), _ptr(d_ssm_state_out), _ptr(d_conv_state_out),
                    _ptr(o["d_ssm_state"]), _ptr(o["d_conv_state"]))
    h = _stream_handle(stream)
    r = raw_bwd_scan(dims, code, _ptr(x), _ptr(delta_raw), _ptr(z), _ptr(Bm), _ptr(Cm),
                     _ptr(conv_w), _ptr(conv_b), _ptr(dt_bias), _ptr(a_log), _ptr(D), _ptr(ckpt),
                     _ptr(d_gated), _ptr(o["du"]), _ptr(o["d_delta_raw"]), _ptr(o["dz"]),
                     o["dB"].data_ptr(), o["dC"].data_ptr(), _ptr(o["d_dt_bias"]),
                     _ptr(o["d_a_log"]), _ptr(o["dD"]), st, ws.ptr, ws.nbytes, h)
    if r != 0:
        raise M3Error(r, "m3scan_bwd_scan")
    du_extra = du_extra_fn(o) if du_extra_fn is not None else None
    if du_extra is not None:
        _check(du_extra, "du_extra", act, dev)
    r = raw_conv_bwd(dims, code, _ptr(x), _ptr(conv_w), _ptr(conv_b), _ptr(o["du"]),
                     _ptr(du_extra), _ptr(o["d_x"]), _ptr(o["d_conv_w"]), _ptr(o["d_conv_b"]),
                     st, ws.ptr, ws.nbytes, h)
    if r != 0:
        raise M3Error(r, "m3scan_conv_bwd")
    return o

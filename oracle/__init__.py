"""CPU oracle for the selective-scan layer core -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``m3scan_oracle.c`` (plain float64 C, single
threaded).  This module compiles it with gcc, loads it with ctypes and wraps
it for NumPy arrays.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the CUDA library never does,
and nothing here imports the CUDA library.

Every function takes the same (already dtype-rounded) inputs the GPU sees,
promoted to float64, and returns float64 results.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3scan_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libm3oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (IEEE float64, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.m3o_forward.restype = ctypes.c_int
            lib.m3o_forward.argtypes = ([_i64] * 5 + [_dp] * 10 + [_u8p] + [_dp] * 5
                                        + [_i64] + [_dp] * 4)
            lib.m3o_backward.restype = ctypes.c_int
            lib.m3o_backward.argtypes = ([_i64] * 5 + [_dp] * 11 + [_u8p, _i64]
                                         + [_dp] * 11 + [_dp] * 7)
            _lib = lib
    return _lib


def _c64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(_dp)


def _opt64(a):
    return None if a is None else _c64(a)


def _mask_ptr(mask):
    if mask is None:
        return None, None
    m = np.ascontiguousarray(np.asarray(mask, dtype=np.uint8))
    return m, m.ctypes.data_as(_u8p)


def _common(inp):
    """Unpack an ``Inputs``-like mapping into float64 arrays and sizes."""
    x = _c64(inp["x"])
    Bsz, T, D = x.shape
    Bm = _c64(inp["B"])
    N = Bm.shape[-1]
    conv_w = _c64(inp["conv_w"])
    W = conv_w.shape[-1]
    arrs = dict(x=x, delta_raw=_c64(inp["delta_raw"]), z=_c64(inp["z"]), B=Bm,
                C=_c64(inp["C"]), conv_w=conv_w, conv_b=_c64(inp["conv_b"]),
                dt_bias=_c64(inp["dt_bias"]), a_log=_c64(inp["a_log"]),
                D=_c64(inp["D"]))
    return (Bsz, T, D, N, W), arrs


def forward(inp, chan_mask=None, ckpt_chunk: int = 0, ssm_state=None, conv_state=None):
    """Oracle forward.

    Returns a dict with ``gated``, ``y``, ``u``, ``delta`` ([B,T,D]),
    ``ssm_state_out`` ([B,N,D], the state after the last step) and
    ``conv_state_out`` ([B,W-1,D], the conv inputs of the last W-1 steps,
    oldest first) and, if ``ckpt_chunk`` > 0, ``ckpt`` ([B, ceil(T/K), N, D],
    the state before each chunk).  ``ssm_state`` ([B,N,D]) and
    ``conv_state`` ([B,W-1,D]) are the carried state the sequence starts
    from (None = zero).  Channels outside ``chan_mask`` are left as zeros.
    """
    lib = _load()
    (Bsz, T, D, N, W), a = _common(inp)
    h0 = _opt64(ssm_state)
    c0 = _opt64(conv_state)
    h_out = np.zeros((Bsz, N, D))
    c_out = np.zeros((Bsz, W - 1, D))
    gated = np.zeros((Bsz, T, D))
    y = np.zeros((Bsz, T, D))
    u = np.zeros((Bsz, T, D))
    delta = np.zeros((Bsz, T, D))
    ckpt = None
    if ckpt_chunk > 0:
        nc = (T + ckpt_chunk - 1) // ckpt_chunk
        ckpt = np.zeros((Bsz, nc, N, D))
    _m, mp = _mask_ptr(chan_mask)
    rc = lib.m3o_forward(Bsz, T, D, N, W, _ptr(a["x"]), _ptr(a["delta_raw"]),
                         _ptr(a["z"]), _ptr(a["B"]), _ptr(a["C"]),
                         _ptr(a["conv_w"]), _ptr(a["conv_b"]), _ptr(a["dt_bias"]),
                         _ptr(a["a_log"]), _ptr(a["D"]), mp, _ptr(gated), _ptr(y),
                         _ptr(u), _ptr(delta), _ptr(ckpt), int(ckpt_chunk),
                         _ptr(h0), _ptr(c0), _ptr(h_out), _ptr(c_out))
    if rc != 0:
        raise MemoryError("oracle forward: allocation failed")
    out = dict(gated=gated, y=y, u=u, delta=delta, ssm_state_out=h_out,
               conv_state_out=c_out)
    if ckpt is not None:
        out["ckpt"] = ckpt
    return out


GRAD_NAMES = ("d_x", "d_delta_raw", "dz", "du", "dB", "dC", "d_conv_w",
              "d_conv_b", "d_dt_bias", "d_a_log", "dD")


STATE_GRAD_NAMES = ("d_ssm_state", "d_conv_state")


def backward(inp, d_gated=None, chan_mask=None, chunk: int = 0, ssm_state=None,
             conv_state=None, d_ssm_state_out=None, d_conv_state_out=None, d_u_extra=None):
    """Oracle backward of
    L = sum(gated * d_gated) + sum(ssm_state_out * d_ssm_state_out)
        + sum(conv_state_out * d_conv_state_out) + sum(u * d_u_extra).

    ``d_u_extra`` [B,T,D] is a gradient reaching u from outside the layer
    core (the x_proj path); ``du`` stays dL/du through the D skip and the
    recurrence only.

    ``chunk`` = 0 keeps every state (sequential); ``chunk`` > 0 recomputes
    states chunk by chunk from chunk-start states.  The carried-state
    arguments are as in ``forward`` (None = zero).  Returns a dict of float64
    gradients named as in ``GRAD_NAMES`` and ``STATE_GRAD_NAMES``.
    """
    lib = _load()
    (Bsz, T, D, N, W), a = _common(inp)
    g = _c64(inp["d_gated"] if d_gated is None else d_gated)
    h0, c0 = _opt64(ssm_state), _opt64(conv_state)
    gh, gc = _opt64(d_ssm_state_out), _opt64(d_conv_state_out)
    gu = _opt64(d_u_extra)
    out = {k: np.zeros((Bsz, T, D)) for k in ("d_x", "d_delta_raw", "dz", "du")}
    out["dB"] = np.zeros((Bsz, T, N))
    out["dC"] = np.zeros((Bsz, T, N))
    out["d_conv_w"] = np.zeros((D, W))
    out["d_conv_b"] = np.zeros(D)
    out["d_dt_bias"] = np.zeros(D)
    out["d_a_log"] = np.zeros((D, N))
    out["dD"] = np.zeros(D)
    out["d_ssm_state"] = np.zeros((Bsz, N, D))
    out["d_conv_state"] = np.zeros((Bsz, W - 1, D))
    _m, mp = _mask_ptr(chan_mask)
    rc = lib.m3o_backward(Bsz, T, D, N, W, _ptr(a["x"]), _ptr(a["delta_raw"]),
                          _ptr(a["z"]), _ptr(a["B"]), _ptr(a["C"]),
                          _ptr(a["conv_w"]), _ptr(a["conv_b"]), _ptr(a["dt_bias"]),
                          _ptr(a["a_log"]), _ptr(a["D"]), _ptr(g), mp, int(chunk),
                          *[_ptr(out[k]) for k in GRAD_NAMES],
                          _ptr(h0), _ptr(c0), _ptr(gh), _ptr(gc),
                          _ptr(out["d_ssm_state"]), _ptr(out["d_conv_state"]), _ptr(gu))
    if rc != 0:
        raise MemoryError("oracle backward: allocation failed")
    return out


def loss(inp, d_gated=None, ssm_state=None, conv_state=None, d_ssm_state_out=None,
         d_conv_state_out=None, d_u_extra=None) -> float:
    """The scalar whose gradient ``backward`` gives (see ``backward``)."""
    g = _c64(inp["d_gated"] if d_gated is None else d_gated)
    f = forward(inp, ssm_state=ssm_state, conv_state=conv_state)
    L = float(np.sum(f["gated"] * g))
    if d_ssm_state_out is not None:
        L += float(np.sum(f["ssm_state_out"] * _c64(d_ssm_state_out)))
    if d_conv_state_out is not None:
        L += float(np.sum(f["conv_state_out"] * _c64(d_conv_state_out)))
    if d_u_extra is not None:
        L += float(np.sum(f["u"] * _c64(d_u_extra)))
    return L


# ---------------------------------------------------------------------------
# All-core timing driver (m3scan_oracle_par.c): the same oracle on every host
# core, one block of channels per OpenMP thread.  Used by the benchmark's
# CPU baseline; the tests compare it with the single-threaded functions above.
# ---------------------------------------------------------------------------

_PAR_SRC = os.path.join(_HERE, "m3scan_oracle_par.c")
_PAR_LIB_PATH = os.path.join(_BUILD_DIR, "libm3oracle_par.so")
_par_lib = None


def build_par(force: bool = False) -> str:
    """Compile the all-core driver (the oracle source included unchanged,
    same float64 flags, plus OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_PAR_SRC))
    if not force and os.path.exists(_PAR_LIB_PATH) and os.path.getmtime(_PAR_LIB_PATH) >= newest:
        return _PAR_LIB_PATH
    tmp = _PAR_LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-fopenmp", "-I", _HERE, "-o", tmp, _PAR_SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _PAR_LIB_PATH)
    return _PAR_LIB_PATH


def _load_par():
    global _par_lib
    with _lock:
        if _par_lib is None:
            lib = ctypes.CDLL(build_par())
            lib.m3o_fwd_bwd_par.restype = ctypes.c_int
            lib.m3o_fwd_bwd_par.argtypes = ([_i64] * 5 + [_dp] * 11 + [ctypes.c_int] + [_dp] * 11
                                            + [ctypes.POINTER(ctypes.c_int)])
            _par_lib = lib
    return _par_lib


def forward_backward_all_cores(inp, threads: int = 0):
    """Forward ``gated`` and the backward of L = sum(gated * d_gated) (no
    carried state) on ``threads`` OpenMP threads (0 = all cores).  Returns
    (dict of float64 arrays named as in ``forward``/``backward``, threads
    used)."""
    lib = _load_par()
    (Bsz, T, D, N, W), a = _common(inp)
    g = _c64(inp["d_gated"])
    out = {k: np.zeros((Bsz, T, D)) for k in ("gated", "d_x", "d_delta_raw", "dz")}
    out["dB"] = np.zeros((Bsz, T, N))
    out["dC"] = np.zeros((Bsz, T, N))
    out["d_conv_w"] = np.zeros((D, W))
    out["d_conv_b"] = np.zeros(D)
    out["d_dt_bias"] = np.zeros(D)
    out["d_a_log"] = np.zeros((D, N))
    out["dD"] = np.zeros(D)
    used = ctypes.c_int(0)
    rc = lib.m3o_fwd_bwd_par(Bsz, T, D, N, W, _ptr(a["x"]), _ptr(a["delta_raw"]), _ptr(a["z"]),
                             _ptr(a["B"]), _ptr(a["C"]), _ptr(a["conv_w"]), _ptr(a["conv_b"]),
                             _ptr(a["dt_bias"]), _ptr(a["a_log"]), _ptr(a["D"]), _ptr(g),
                             int(threads), _ptr(out["gated"]), _ptr(out["d_x"]),
                             _ptr(out["d_delta_raw"]), _ptr(out["dz"]), _ptr(out["dB"]),
                             _ptr(out["dC"]), _ptr(out["d_conv_w"]), _ptr(out["d_conv_b"]),
                             _ptr(out["d_dt_bias"]), _ptr(out["d_a_log"]), _ptr(out["dD"]),
                             ctypes.byref(used))
    if rc != 0:
        raise MemoryError("oracle (all cores): allocation failed")
    return out, int(used.value)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))

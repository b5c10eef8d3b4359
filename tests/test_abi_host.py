"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/m3scan.h declares, and its
argument validation rejects bad calls before anything is enqueued.

Every call here that passes addresses is built to fail validation (NULL,
misaligned, unsupported or undersized arguments), so nothing ever reaches a
device even where one is present.
"""

import ctypes
import os
import re

import pytest

from mamba_selective_scan_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "m3scan.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(m3scan_\w+)\s*\(", src)))


def test_header_declares_what_the_binding_exports():
    assert _declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert binding.m3scan_version() == 10100  # 1.1.0
    for code, name in binding.STATUS.items():
        assert binding.m3scan_status_string(code).startswith(name)
    assert "unknown" in binding.m3scan_status_string(99)


def _plan(dims, act=binding.M3_BF16):
    out = binding.M3Plan()
    st = binding.load().m3scan_plan(ctypes.byref(dims), act, ctypes.byref(out))
    return st, out


def test_plan_with_explicit_segments_needs_no_device(lib):
    dims = binding.make_dims(8, 2048, 1536, chunk=16, segments=4)
    st, p = _plan(dims)
    assert st == 0
    assert p.chunk == 16 and p.n_chunks == 128
    assert p.fwd_segments == 4 and p.bwd_segments == 4
    assert p.ckpt_bytes == 8 * 128 * 16 * 1536 * 4
    # 8 x 12 x 4 blocks fit one wave: the split kernels, whose backward main
    # kernel finishes the parameter gradients itself (aggregate + main)
    assert p.bwd_threads_per_channel == 2
    assert p.fwd_launches == 2 and p.bwd_launches == 2
    # the one-thread kernels: aggregate + main + parameter-gradient tail
    st, pt = _plan(binding.make_dims(8, 2048, 1536, chunk=16, segments=4, threads_per_channel=1))
    assert st == 0 and pt.bwd_launches == 3
    assert pt.workspace_bytes >= 8 * 4 * 24 * 1536 * 4
    # deterministic: the tail kernel and the dB/dC sum kernel as well
    st, pd = _plan(binding.make_dims(8, 2048, 1536, chunk=16, segments=4, deterministic=True))
    assert st == 0 and pd.bwd_launches == 4
    # one segment: the main kernel plus the parameter-gradient tail kernel
    st, p1 = _plan(binding.make_dims(8, 2048, 1536, chunk=16, segments=1))
    assert st == 0 and p1.fwd_launches == 1 and p1.bwd_launches == 2
    assert p1.workspace_bytes >= 8 * 24 * 1536 * 4


def test_segments_are_whole_chunks_of_at_least_four_steps(lib):
    st, p = _plan(binding.make_dims(1, 10, 8, chunk=1, segments=10))
    assert st == 0
    # chunk 1 -> at least 4 chunks per segment -> ceil(10 / 4) = 3 segments
    assert p.fwd_segments == 3 and p.bwd_segments == 3
    st, p = _plan(binding.make_dims(1, 10, 8, chunk=16, segments=7))
    assert st == 0 and p.fwd_segments == 1


@pytest.mark.parametrize("kw,status", [
    (dict(d_state=8), "M3_ERR_UNSUPPORTED"),
    (dict(d_conv=3), "M3_ERR_UNSUPPORTED"),
    (dict(d_inner=36), "M3_ERR_UNSUPPORTED"),
    (dict(batch=-1), "M3_ERR_DIMS"),
    (dict(seq_len=-5), "M3_ERR_DIMS"),
    (dict(chunk=257), "M3_ERR_DIMS"),
    (dict(chunk=60), "M3_ERR_UNSUPPORTED"),  # longer than a tile, not a whole number of tiles
    (dict(segments=-1), "M3_ERR_DIMS"),
    (dict(batch=70000), "M3_ERR_DIMS"),
])
def test_plan_rejects_bad_dims(lib, kw, status):
    base = dict(batch=2, seq_len=64, d_inner=64, d_state=16, d_conv=4, chunk=16, segments=1)
    base.update(kw)
    st, _ = _plan(binding.make_dims(**base))
    assert binding.STATUS[st] == status


def test_plan_rejects_unknown_dtype_and_null(lib):
    st, _ = _plan(binding.make_dims(1, 8, 8, segments=1), act=7)
    assert binding.STATUS[st] == "M3_ERR_UNSUPPORTED"
    assert binding.STATUS[lib.m3scan_plan(None, 1, None)] == "M3_ERR_NULL"


def test_chunk_is_up_to_a_tile_or_whole_tiles_up_to_256(lib):
    def st(chunk, act=binding.M3_BF16):
        return binding.STATUS[_plan(binding.make_dims(1, 64, 64, chunk=chunk, segments=1), act)[0]]
    for k in (1, 5, 7, 8, 16, 24, 64, 128, 256):
        assert st(k) == "M3_OK" and st(k, binding.M3_F32) == "M3_OK", k
    for k in (9, 30, 63, 100, 250):
        assert st(k) == "M3_ERR_UNSUPPORTED", k
    assert st(264) == "M3_ERR_DIMS"


def test_default_chunk(lib):
    for T in (128, 1024, 65536):
        _, pl = _plan(binding.make_dims(1, T, 64, segments=1))
        assert pl.chunk == 8, T


def test_long_chunks_add_sub_checkpoints_to_the_workspace(lib):
    """Per block of the backward's main kernel: the states before tiles
    1 .. K/8 - 2 of its chunk (16 floats x 128 channels each)."""
    def ws(chunk, segments=3):
        _, pl = _plan(binding.make_dims(2, 1024, 256, chunk=chunk, segments=segments,
                                        threads_per_channel=1))
        return pl.workspace_bytes, pl
    small, _ = ws(16)      # two tiles: none kept
    big, pl = ws(64)       # eight tiles: six kept
    blocks = 2 * 3 * 2     # channel blocks x segments x batch
    sub = blocks * 6 * 16 * 128 * 4
    assert small < sub <= big
    assert pl.chunk == 64 and pl.n_chunks == 16


A = 1 << 20  # a 256-byte aligned fake address; never dereferenced


def _fwd_args(**over):
    a = dict(x=A, delta_raw=A, z=A, Bm=A, Cm=A, conv_w=A, conv_b=A, dt_bias=A, a_log=A,
             D=A, gated=A, y_dbg=None, ckpt=A, workspace=A, workspace_bytes=1 << 30,
             stream=None)
    a.update(over)
    return a


def _fwd(dims, act=binding.M3_BF16, **over):
    a = _fwd_args(**over)
    return binding.STATUS[binding.raw_fwd(dims, act, a["x"], a["delta_raw"], a["z"], a["Bm"],
                                          a["Cm"], a["conv_w"], a["conv_b"], a["dt_bias"],
                                          a["a_log"], a["D"], a["gated"], a["y_dbg"],
                                          a["ckpt"], a["workspace"], a["workspace_bytes"],
                                          a["stream"])]


def test_fwd_rejects_null_and_misaligned_before_any_launch(lib):
    dims = binding.make_dims(2, 64, 64, chunk=16, segments=2)
    assert _fwd(dims, x=None) == "M3_ERR_NULL"
    assert _fwd(dims, ckpt=None) == "M3_ERR_NULL"
    assert _fwd(dims, gated=None) == "M3_ERR_NULL"
    assert _fwd(dims, x=A + 2) == "M3_ERR_ALIGN"
    assert _fwd(dims, Cm=A + 8) == "M3_ERR_ALIGN"
    assert _fwd(dims, y_dbg=A + 4) == "M3_ERR_ALIGN"
    assert _fwd(dims, conv_w=A + 1) == "M3_ERR_ALIGN"
    assert _fwd(dims, workspace=None) == "M3_ERR_WORKSPACE"
    assert _fwd(dims, workspace_bytes=16) == "M3_ERR_WORKSPACE"
    assert _fwd(dims, workspace=A + 16) == "M3_ERR_ALIGN"
    assert _fwd(binding.make_dims(2, 64, 60, segments=1)) == "M3_ERR_UNSUPPORTED"


def test_empty_forward_is_a_no_op(lib):
    # zero elements: nothing to do, nothing is touched, pointers may be NULL
    dims = binding.make_dims(0, 64, 64, segments=1)
    assert _fwd(dims, x=None, gated=None, ckpt=None) == "M3_OK"


def _bwd(dims, act=binding.M3_BF16, **over):
    a = dict(x=A, delta_raw=A, z=A, Bm=A, Cm=A, conv_w=A, conv_b=A, dt_bias=A, a_log=A, D=A,
             ckpt=A, d_gated=A, d_x=A, d_delta_raw=A, dz=A, du_dbg=None, dB=A, dC=A,
             d_conv_w=A, d_conv_b=A, d_dt_bias=A, d_a_log=A, dD=A, workspace=A,
             workspace_bytes=1 << 30, stream=None)
    a.update(over)
    return binding.STATUS[binding.raw_bwd(dims, act, *a.values())]


def test_bwd_rejects_bad_arguments_before_any_launch(lib):
    dims = binding.make_dims(2, 64, 64, chunk=16, segments=1)
    assert _bwd(dims, d_gated=None) == "M3_ERR_NULL"
    assert _bwd(dims, dB=None) == "M3_ERR_NULL"
    assert _bwd(dims, dD=None) == "M3_ERR_NULL"
    assert _bwd(dims, d_x=A + 2) == "M3_ERR_ALIGN"
    assert _bwd(dims, du_dbg=A + 2) == "M3_ERR_ALIGN"
    assert _bwd(dims, dC=A + 2) == "M3_ERR_ALIGN"
    assert _bwd(dims, workspace=None) == "M3_ERR_WORKSPACE"
    assert _bwd(dims, workspace_bytes=255) == "M3_ERR_WORKSPACE"
    assert _bwd(dims, workspace=A + 128) == "M3_ERR_ALIGN"
    assert _bwd(binding.make_dims(2, 64, 64, d_state=24, segments=1)) == "M3_ERR_UNSUPPORTED"
    # wider states run on the split kernels only
    assert _bwd(binding.make_dims(2, 64, 64, d_state=32, segments=1,
                                  threads_per_channel=1)) == "M3_ERR_UNSUPPORTED"


def _fwd_state(dims, state, act=binding.M3_BF16, **over):
    a = dict(x=A, delta_raw=A, z=A, Bm=A, Cm=A, conv_w=A, conv_b=A, dt_bias=A, a_log=A, D=A,
             gated=A, y_dbg=None, ckpt=A)
    a.update(over)
    return binding.STATUS[binding.raw_fwd_state(dims, act, *a.values(), state, A, 1 << 30,
                                                None)]


def _bwd_state(dims, state, act=binding.M3_BF16):
    a = dict(x=A, delta_raw=A, z=A, Bm=A, Cm=A, conv_w=A, conv_b=A, dt_bias=A, a_log=A, D=A,
             ckpt=A, d_gated=A, d_x=A, d_delta_raw=A, dz=A, du_dbg=None, dB=A, dC=A,
             d_conv_w=A, d_conv_b=A, d_dt_bias=A, d_a_log=A, dD=A)
    return binding.STATUS[binding.raw_bwd_state(dims, act, *a.values(), state, A, 1 << 30, None)]


def test_state_entry_points_validate_before_any_launch(lib):
    dims = binding.make_dims(2, 64, 64, chunk=16, segments=2)
    # the state struct itself is required by the _state entry points
    assert _fwd_state(dims, None) == "M3_ERR_NULL"
    assert _bwd_state(dims, None) == "M3_ERR_NULL"
    # float32 state 4-byte aligned, activation-dtype state aligned to its element
    assert _fwd_state(dims, binding.M3FwdState(A + 2, None, None, None)) == "M3_ERR_ALIGN"
    assert _fwd_state(dims, binding.M3FwdState(None, None, None, A + 1)) == "M3_ERR_ALIGN"
    assert _fwd_state(dims, binding.M3FwdState(None, A + 2, None, None),
                      act=binding.M3_F32) == "M3_ERR_ALIGN"
    assert _bwd_state(dims, binding.M3BwdState(None, A + 2, None, None, None)) == "M3_ERR_ALIGN"
    assert _bwd_state(dims, binding.M3BwdState(None, None, None, None, A + 1)) == "M3_ERR_ALIGN"
    # the other arguments are still checked
    assert _fwd_state(dims, binding.M3FwdState(A, A + 2, A, A + 2), x=None) == "M3_ERR_NULL"


def test_state_structs_match_the_header_layout():
    assert ctypes.sizeof(binding.M3FwdState) == 4 * ctypes.sizeof(ctypes.c_void_p)
    assert ctypes.sizeof(binding.M3BwdState) == 5 * ctypes.sizeof(ctypes.c_void_p)
    src = open(os.path.join(ROOT, "include", "m3scan.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for struct, cls in (("m3_fwd_state", binding.M3FwdState), ("m3_bwd_state", binding.M3BwdState)):
        body = re.search(r"typedef struct \{([^{}]*)\}\s*" + struct + ";", src).group(1)
        names = re.findall(r"(\w+);", body)
        assert names == [f for f, _ in cls._fields_], struct


def _decode(dims, act=binding.M3_BF16, **over):
    a = dict(x=A, delta_raw=A, z=A, Bm=A, Cm=A, conv_w=A, conv_b=A, dt_bias=A, a_log=A, D=A,
             ssm_state=A, conv_state=A, gated=A, y_dbg=None, stream=None)
    a.update(over)
    return binding.STATUS[binding.raw_decode(dims, act, *a.values())]


def test_decode_validates_before_any_launch(lib):
    for n in (16, 32, 64):
        assert _decode(binding.make_dims(2, 1, 64, d_state=n), x=None) == "M3_ERR_NULL"
    assert _decode(binding.make_dims(2, 1, 64, d_state=24)) == "M3_ERR_UNSUPPORTED"
    assert _decode(binding.make_dims(2, 1, 64, d_state=128)) == "M3_ERR_UNSUPPORTED"
    assert _decode(binding.make_dims(2, 1, 64, d_conv=3)) == "M3_ERR_UNSUPPORTED"
    assert _decode(binding.make_dims(2, 1, 64), act=7) == "M3_ERR_UNSUPPORTED"
    assert _decode(binding.make_dims(-1, 1, 64)) == "M3_ERR_DIMS"
    assert _decode(binding.make_dims(2, 1, 64), ssm_state=None) == "M3_ERR_NULL"
    assert _decode(binding.make_dims(2, 1, 64), conv_state=None) == "M3_ERR_NULL"
    assert _decode(binding.make_dims(2, 1, 64), ssm_state=A + 2) == "M3_ERR_ALIGN"
    assert _decode(binding.make_dims(2, 1, 64), x=A + 1) == "M3_ERR_ALIGN"
    assert _decode(binding.make_dims(2, 1, 64), x=A + 2, act=binding.M3_F32) == "M3_ERR_ALIGN"
    # element alignment is enough for bf16; any d_inner is accepted
    assert _decode(binding.make_dims(2, 0, 60), x=A + 2) == "M3_OK"
    # nothing to do: no pointer is needed
    assert _decode(binding.make_dims(2, 0, 64), x=None, ssm_state=None) == "M3_OK"


def _struct_fields(name):
    src = open(os.path.join(ROOT, "include", "m3scan.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = re.search(r"typedef struct \{([^{}]*)\}\s*" + name + ";", src).group(1)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        parts = decl.split(",")
        names.append(re.findall(r"(\w+)\s*$", parts[0])[0])
        names += [p.strip() for p in parts[1:]]
    return names


def test_dims_and_plan_structs_match_the_header():
    assert _struct_fields("m3_dims") == [f for f, _ in binding.M3Dims._fields_]
    assert _struct_fields("m3_plan") == [f for f, _ in binding.M3Plan._fields_]
    assert ctypes.sizeof(binding.M3Dims) == 8 * 7 + 4 * 2 + 8 * 2 + 4 * 2


def test_row_strides_are_validated(lib):
    out = binding.M3Plan()
    def plan(**kw):
        d = binding.make_dims(2, 64, 64, segments=1, **kw)
        return binding.STATUS[lib.m3scan_plan(ctypes.byref(d), binding.M3_BF16, ctypes.byref(out))]
    assert plan(bc_stride=48, dbc_stride=48) == "M3_OK"      # dt_rank 16 + 2 x 16
    assert plan(bc_stride=8) == "M3_ERR_DIMS"                 # narrower than d_state
    assert plan(dbc_stride=15) == "M3_ERR_DIMS"
    assert plan(bc_stride=-16) == "M3_ERR_DIMS"
    assert plan(bc_stride=20) == "M3_ERR_ALIGN"               # 40 bytes: not a multiple of 16
    assert plan(dbc_stride=17) == "M3_OK"                     # dB/dC take any stride


def test_two_phase_entry_points_validate_before_any_launch(lib):
    dims = binding.make_dims(2, 64, 64, chunk=16, segments=2)
    a = dict(x=A, delta_raw=A, z=A, Bm=A, Cm=A, conv_w=A, conv_b=A, dt_bias=A, a_log=A, D=A,
             ckpt=A, d_gated=A, du=A, d_delta_raw=A, dz=A, dB=A, dC=A, d_dt_bias=A, d_a_log=A,
             dD=A)
    def scan(**over):
        b = dict(a)
        b.update(over)
        return binding.STATUS[binding.raw_bwd_scan(dims, binding.M3_BF16, *b.values(), None, A,
                                                   1 << 30, None)]
    assert scan(du=None) == "M3_ERR_NULL"
    assert scan(dD=None) == "M3_ERR_NULL"
    assert scan(du=A + 2) == "M3_ERR_ALIGN"
    def conv(**over):
        c = dict(x=A, conv_w=A, conv_b=A, du=A, du_extra=None, d_x=A, d_conv_w=A, d_conv_b=A)
        c.update(over)
        ws = c.pop("ws", 1 << 30)
        return binding.STATUS[binding.raw_conv_bwd(dims, binding.M3_BF16, *c.values(), None, A,
                                                   ws, None)]
    assert conv(du=None) == "M3_ERR_NULL"
    assert conv(d_x=None) == "M3_ERR_NULL"
    assert conv(du_extra=A + 2) == "M3_ERR_ALIGN"
    assert conv(ws=16) == "M3_ERR_WORKSPACE"


def test_threads_per_channel_are_resolved_from_the_grid(lib):
    def tpc(batch, T, D, seg, want=0, chunk=8):
        out = binding.M3Plan()
        d = binding.make_dims(batch, T, D, chunk=chunk, segments=seg, threads_per_channel=want)
        st = lib.m3scan_plan(ctypes.byref(d), binding.M3_BF16, ctypes.byref(out))
        return binding.STATUS[st] if st else (out.fwd_threads_per_channel,
                                              out.bwd_threads_per_channel)
    # grids under one wave of the one-thread kernels (6 forward, 3 backward
    # blocks per SM of a 152-SM GPU) take two threads per channel
    assert tpc(8, 128, 512, 8) == (2, 2)            # 8 x 4 groups x 8 segments = 256 blocks
    assert tpc(8, 2048, 1536, 12) == (1, 1)         # 8 x 12 x 12 = 1152 blocks
    assert tpc(8, 2048, 1536, 6) == (2, 1)          # 576 blocks: one forward wave, not backward
    assert tpc(8, 2048, 1536, 12, want=2) == (2, 2)  # an explicit choice wins
    assert tpc(8, 128, 512, 8, want=1) == (1, 1)
    assert tpc(8, 128, 512, 8, want=3) == "M3_ERR_UNSUPPORTED"


def test_wider_states_resolve_to_the_split_kernels(lib):
    for n, tpc in ((32, 4), (64, 8)):
        out = binding.M3Plan()
        d = binding.make_dims(2, 256, 512, d_state=n, chunk=8, segments=2)
        assert lib.m3scan_plan(ctypes.byref(d), binding.M3_BF16, ctypes.byref(out)) == 0
        assert (out.fwd_threads_per_channel, out.bwd_threads_per_channel) == (tpc, tpc)
        assert out.ckpt_bytes == 2 * 32 * n * 512 * 4


def test_device_status_rejects_null(lib):
    assert lib.m3scan_device_status(None) == 1  # M3_ERR_NULL


def test_get_status_rejects_null_and_misaligned_before_touching_a_device(lib):
    out = ctypes.c_int(0)
    assert binding.STATUS[lib.m3scan_get_status(None, None, ctypes.byref(out))] == "M3_ERR_NULL"
    assert binding.STATUS[lib.m3scan_get_status(1 << 20, None, None)] == "M3_ERR_NULL"
    assert binding.STATUS[lib.m3scan_get_status((1 << 20) + 16, None, ctypes.byref(out))] == \
        "M3_ERR_ALIGN"
    assert binding.STATUS[lib.m3scan_selftest_wait_timeout((1 << 20) + 16, None)] == "M3_ERR_ALIGN"


def test_workspace_begins_with_the_status_block(lib):
    """Every section of the workspace starts after the status block, and the
    smallest workspace holds it."""
    dims = binding.make_dims(1, 8, 8, chunk=8, segments=1)
    pl = binding.m3scan_plan(dims, binding.M3_F32)
    assert pl.workspace_bytes >= binding.STATUS_BYTES == 256


def test_deterministic_adds_block_partials_to_the_workspace(lib):
    base = binding.make_dims(8, 2048, 1536, chunk=8, segments=12, threads_per_channel=1)
    det = binding.make_dims(8, 2048, 1536, chunk=8, segments=12, threads_per_channel=1,
                            deterministic=True)
    st0, p0 = _plan(base)
    st1, p1 = _plan(det)
    assert st0 == 0 and st1 == 0
    # 12 blocks of 128 channels, one partial row of 2 x 16 floats per (batch, step, block)
    assert p1.workspace_bytes >= p0.workspace_bytes + 8 * 2048 * 12 * 32 * 4 - 256
    bad = binding.make_dims(8, 2048, 1536, chunk=8, segments=12)
    bad.deterministic = 2
    assert binding.STATUS[_plan(bad)[0]] == "M3_ERR_DIMS"
    bad = binding.make_dims(8, 2048, 1536, chunk=8, segments=12)
    bad.reserved0 = 1
    assert binding.STATUS[_plan(bad)[0]] == "M3_ERR_DIMS"


def test_cluster_finish_covers_two_to_eight_backward_segments(lib):
    """The split backward finishes its sums in a cluster of its segments when
    there are 2-8 of them (aggregate + main kernel, no partials region);
    with more segments, one thread per channel, or deterministic sums the
    tail kernel runs after it."""
    def plan(**kw):
        st, p = _plan(binding.make_dims(2, 1024, 256, chunk=8, **kw))
        assert st == 0
        return p
    p8 = plan(segments=8, threads_per_channel=2)
    assert p8.bwd_segments == 8 and p8.bwd_launches == 2
    p9 = plan(segments=9, threads_per_channel=2)
    assert p9.bwd_segments == 9 and p9.bwd_launches == 3
    # the cluster path needs no per-(batch, segment) partials [B * S, N + 8, D]
    assert p9.workspace_bytes >= p8.workspace_bytes + 2 * 8 * 24 * 256 * 4 - 256 * 8
    assert plan(segments=8, threads_per_channel=1).bwd_launches == 3
    assert plan(segments=8, threads_per_channel=2, deterministic=True).bwd_launches == 4
    assert plan(segments=1, threads_per_channel=2).bwd_launches == 2  # main + tail

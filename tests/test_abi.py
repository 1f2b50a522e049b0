"""C-ABI checks that need no GPU: the library loads, exports every function
include/vsa.h declares, and vsa_plan_create validates shapes on the host."""
import ctypes
import os

import pytest

import block_sparse_video_gb300 as bsv
from block_sparse_video_gb300.synthetic import CONFIGS
from oracle import vsa_oracle as vo


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bsv.LIB_PATH):
        from block_sparse_video_gb300 import build
        build.build()
    return bsv.load_library()


def test_exports_every_declared_function(lib):
    names = bsv.header_functions()
    assert {"vsa_plan_create", "vsa_plan_info", "vsa_forward", "vsa_forward_host", "vsa_check",
            "vsa_debug_views", "vsa_plan_destroy", "vsa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def _status(**kw):
    shape = dict(batch=1, num_heads=2, head_dim=128, len_text=64, len_audio=64, len_video=1024,
                 keep_fraction=0.2)
    shape.update(kw)
    s = bsv.vsa_shape_t(shape["batch"], shape["num_heads"], shape["head_dim"], shape["len_text"],
                        shape["len_audio"], shape["len_video"], shape["keep_fraction"])
    out = ctypes.c_void_p()
    st = bsv.load_library().vsa_plan_create(ctypes.byref(s), 0, ctypes.byref(out))
    if out.value:
        bsv.vsa_plan_destroy(out.value)
    return st


def test_plan_validation_status_codes(lib):
    assert _status() == bsv.VSA_OK
    assert _status(head_dim=64) == bsv.VSA_ERR_UNSUPPORTED
    assert _status(len_video=0) == bsv.VSA_ERR_INVALID_ARG
    assert _status(len_text=-1) == bsv.VSA_ERR_INVALID_ARG
    assert _status(batch=0) == bsv.VSA_ERR_INVALID_ARG
    assert _status(num_heads=0) == bsv.VSA_ERR_INVALID_ARG
    for f in (0.0, -0.1, 1.5, float("nan"), float("inf")):
        assert _status(keep_fraction=f) == bsv.VSA_ERR_INVALID_ARG, f
    assert _status(len_video=1 << 30) == bsv.VSA_ERR_UNSUPPORTED
    assert _status(len_text=0, len_audio=0) == bsv.VSA_OK  # empty prefix is allowed
    assert _status(len_video=1) == bsv.VSA_OK
    assert _status(keep_fraction=1.0) == bsv.VSA_OK
    assert lib.vsa_plan_create(None, 0, None) == bsv.VSA_ERR_INVALID_ARG


def test_plan_counts_match_oracle(lib):
    cases = [(c.len_video, f) for c in CONFIGS.values() for f in c.keep]
    cases += [(1, 0.2), (64, 0.2), (65, 0.2), (320, 0.5), (640, 0.25), (448, 1.0), (192, 0.01)]
    for lv, f in cases:
        plan = bsv.vsa_plan_create(1, 1, 10, 20, lv, f)
        try:
            t, k, ws = bsv.vsa_plan_info(plan)
        finally:
            bsv.vsa_plan_destroy(plan)
        assert t == vo.video_tile_count(lv)
        assert k == vo.keep_count(t, f), (lv, f)
        assert ws >= 256 + 4 * t * 128 * 4 + t * k * 4


def test_forward_rejects_bad_arguments_without_launching(lib):
    plan = bsv.vsa_plan_create(1, 2, 64, 64, 1024, 0.2)
    try:
        _, _, ws = bsv.vsa_plan_info(plan)
        f = lib.vsa_forward
        fake = ctypes.c_void_p(1 << 20)
        assert f(plan, None, fake, fake, fake, fake, fake, ws, None) == bsv.VSA_ERR_INVALID_ARG
        # workspace too small
        assert f(plan, fake, fake, fake, fake, fake, fake, ws - 1, None) == bsv.VSA_ERR_INVALID_ARG
        # misaligned input
        a = ctypes.c_void_p((1 << 30) + 8)
        assert f(plan, a, fake, fake, fake, ctypes.c_void_p(1 << 34), ctypes.c_void_p(1 << 36), ws,
                 None) == bsv.VSA_ERR_INVALID_ARG
        # out aliasing an input
        x = ctypes.c_void_p(1 << 30)
        assert f(plan, x, ctypes.c_void_p(1 << 31), ctypes.c_void_p(1 << 32), ctypes.c_void_p(1 << 33), x,
                 ctypes.c_void_p(1 << 36), ws, None) == bsv.VSA_ERR_INVALID_ARG
        assert lib.vsa_check(None, fake, None) == bsv.VSA_ERR_INVALID_ARG
    finally:
        bsv.vsa_plan_destroy(plan)


def test_status_strings(lib):
    for s in range(6):
        assert bsv.vsa_status_string(s)
    assert "timed out" in bsv.vsa_status_string(bsv.VSA_ERR_DEVICE_TIMEOUT)


def _pre_args(**kw):
    """A vsa_preprocess_args_t with well-formed fake device addresses (never
    dereferenced: every case below is rejected on the host)."""
    g = 1 << 32
    a = dict(q_in=1 * g, k_in=1 * g + 256, v_in=1 * g + 512, gate_in=1 * g + 768, rows_in=2000,
             row_stride=4 * 2 * 128, src_row=None, q_norm_weight=3 * g, k_norm_weight=3 * g + 4096,
             eps=1e-6, rope_dim=96, rope_interleaved=1, rope_cos=4 * g, rope_sin=5 * g,
             q_out=6 * g, k_out=7 * g, v_out=8 * g, gate_out=9 * g)
    a.update(kw)
    return bsv.vsa_preprocess_args_t(**a)


def test_preprocess_rejects_bad_arguments_without_launching(lib):
    plan = bsv.vsa_plan_create(1, 2, 64, 64, 1024, 0.2)  # N = 1152
    try:
        _, _, ws = bsv.vsa_plan_info(plan)
        wsp = ctypes.c_void_p(10 << 32)

        def st(**kw):
            return lib.vsa_preprocess(plan, ctypes.byref(_pre_args(**kw)), wsp, ws, None)

        bad = [
            dict(rows_in=1000),                    # no map and fewer rows than tokens
            dict(rows_in=0, src_row=11 << 32),
            dict(row_stride=2 * 128 - 8),          # shorter than one row of all heads
            dict(row_stride=4 * 2 * 128 + 4),      # not a multiple of 8 elements
            dict(eps=0.0), dict(eps=float("nan")),
            dict(rope_dim=90), dict(rope_dim=144), dict(rope_dim=-16),
            dict(rope_cos=None),
            dict(rope_sin=(5 << 32) + 4),          # misaligned table
            dict(q_norm_weight=None),
            dict(k_in=(1 << 32) + 8),              # misaligned input
            dict(v_out=None),
            dict(gate_out=6 << 32),                # two outputs alias
            dict(q_out=(1 << 32) + 1024),          # output inside the input rows
            dict(src_row=(11 << 32) + 2),          # misaligned map
        ]
        for kw in bad:
            assert st(**kw) == bsv.VSA_ERR_INVALID_ARG, kw
        assert st(row_stride=1 << 25) == bsv.VSA_ERR_UNSUPPORTED
        assert lib.vsa_preprocess(plan, None, wsp, ws, None) == bsv.VSA_ERR_INVALID_ARG
        assert lib.vsa_preprocess(plan, ctypes.byref(_pre_args()), wsp, ws - 1, None) == bsv.VSA_ERR_INVALID_ARG
        # an output overlapping the workspace
        assert lib.vsa_preprocess(plan, ctypes.byref(_pre_args(k_out=10 << 32)), wsp, ws,
                                  None) == bsv.VSA_ERR_INVALID_ARG
        f = lib.vsa_forward_preprocessed
        fake = ctypes.c_void_p(1 << 20)
        assert f(plan, None, fake, fake, fake, fake, fake, ws, None) == bsv.VSA_ERR_INVALID_ARG
    finally:
        bsv.vsa_plan_destroy(plan)


def test_subblock_plan_counts_and_validation(lib):
    from oracle import subblock_oracle as so
    for lv, s in [(72576, 0.75), (72576, 0.8), (36288, 0.75), (1000, 0.5), (50, 0.75), (640, 0.0),
                  (64 * 40, 0.95), (72500, 0.8), (64 * 2600 - 30, 0.8)]:
        plan = bsv.vsa_plan_create_subblock(1, 2, 10, 20, lv, s)
        try:
            t, k, ws = bsv.vsa_plan_info(plan)
        finally:
            bsv.vsa_plan_destroy(plan)
        assert t == vo.video_tile_count(lv)
        assert k == so.keep_count(t, s), (lv, s)
        assert ws >= 256 + 2 * 2 * 4 * t * 128 * 4 + 2 * t * k * 4
    shape = bsv.vsa_shape_t(1, 2, 128, 64, 64, 1024, float("nan"))  # keep_fraction is ignored
    out = ctypes.c_void_p()
    for s in (-0.1, 1.0, float("nan"), float("inf")):
        assert lib.vsa_plan_create_subblock(ctypes.byref(shape), s, 0, ctypes.byref(out)) == bsv.VSA_ERR_INVALID_ARG
    assert lib.vsa_plan_create_subblock(ctypes.byref(shape), 0.75, 0, ctypes.byref(out)) == bsv.VSA_OK
    plan = out.value
    try:
        _, _, ws = bsv.vsa_plan_info(plan)
        fake = ctypes.c_void_p(1 << 20)
        # a VSA plan needs its gate; a SubBlock plan does not (rejected here only for the workspace size)
        vplan = bsv.vsa_plan_create(1, 2, 64, 64, 1024, 0.2)
        try:
            assert lib.vsa_forward(vplan, fake, fake, fake, None, fake, fake, ws, None) == bsv.VSA_ERR_INVALID_ARG
        finally:
            bsv.vsa_plan_destroy(vplan)
        assert lib.vsa_forward(plan, fake, fake, fake, None, fake, fake, ws - 1, None) == bsv.VSA_ERR_INVALID_ARG
    finally:
        bsv.vsa_plan_destroy(plan)
    big = bsv.vsa_shape_t(1, 1, 128, 0, 0, 64 * 20000, 1.0)   # T too large for the router's tiles
    assert lib.vsa_plan_create_subblock(ctypes.byref(big), 0.5, 0, ctypes.byref(out)) == bsv.VSA_ERR_UNSUPPORTED


def test_forward_rows_rejects_bad_layouts_without_launching(lib):
    plan = bsv.vsa_plan_create(1, 2, 64, 64, 1024, 0.2)  # N = 1152, rows of 256 elements
    try:
        _, _, ws = bsv.vsa_plan_info(plan)
        g = 1 << 32
        ins = [ctypes.c_void_p(g * (i + 1)) for i in range(4)]
        wsp = ctypes.c_void_p(10 * g)

        def st(**kw):
            a = dict(out=6 * g, out_rows=2000, out_row_stride=256, out_row_map=None)
            a.update(kw)
            rows = bsv.vsa_output_rows_t(**a)
            return lib.vsa_forward_rows(plan, *ins, ctypes.byref(rows), 0, wsp, ws, None)

        for kw in (dict(out_rows=1000),                    # no map: fewer rows than tokens
                   dict(out_rows=0, out_row_map=11 * g),
                   dict(out_row_stride=255), dict(out_row_stride=252),
                   dict(out_row_map=11 * g + 2),           # misaligned map
                   dict(out=g + 4096),                     # inside an input
                   dict(out=10 * g - 1024),                # running into the workspace
                   dict(out=6 * g + 8)):                   # misaligned output
            assert st(**kw) == bsv.VSA_ERR_INVALID_ARG, kw
        assert st(out_row_stride=1 << 25) == bsv.VSA_ERR_UNSUPPORTED
        assert lib.vsa_forward_rows(plan, *ins, None, 0, wsp, ws, None) == bsv.VSA_ERR_INVALID_ARG
    finally:
        bsv.vsa_plan_destroy(plan)


def test_forward_ex_and_lengths_validation(lib):
    plan = bsv.vsa_plan_create(1, 2, 64, 64, 1024, 0.2)
    sub = bsv.vsa_plan_create_subblock(1, 2, 64, 64, 1024, 0.75)
    try:
        _, _, ws = bsv.vsa_plan_info(plan)
        g = 1 << 32
        wsp = ctypes.c_void_p(10 * g)
        assert lib.vsa_forward_ex(plan, None, wsp, ws, None) == bsv.VSA_ERR_INVALID_ARG
        args = bsv.vsa_forward_args_t(g, 2 * g, 3 * g, 4 * g, 6 * g, None, 12 * g + 4, 0)  # misaligned lengths
        assert lib.vsa_forward_ex(plan, ctypes.byref(args), wsp, ws, None) == bsv.VSA_ERR_INVALID_ARG
        args = bsv.vsa_forward_args_t(g, 2 * g, 3 * g, 4 * g, None, None, None, 0)          # no output
        assert lib.vsa_forward_ex(plan, ctypes.byref(args), wsp, ws, None) == bsv.VSA_ERR_INVALID_ARG
        _, _, ws_sub = bsv.vsa_plan_info(sub)
        args = bsv.vsa_forward_args_t(g, 2 * g, 3 * g, None, 6 * g, None, 12 * g + 4, 0)   # SubBlock, misaligned lengths
        assert lib.vsa_forward_ex(sub, ctypes.byref(args), wsp, ws_sub, None) == bsv.VSA_ERR_INVALID_ARG
        # input row stride: below H x 128, not a multiple of 8, negative; beyond 2^24 is unsupported
        for bad in (255, 260, -8):
            args = bsv.vsa_forward_args_t(g, 2 * g, 3 * g, 4 * g, 6 * g, None, None, 0, bad)
            assert lib.vsa_forward_ex(plan, ctypes.byref(args), wsp, ws, None) == bsv.VSA_ERR_INVALID_ARG, bad
        args = bsv.vsa_forward_args_t(g, 2 * g, 3 * g, 4 * g, 6 * g, None, None, 0, (1 << 24) + 8)
        assert lib.vsa_forward_ex(plan, ctypes.byref(args), wsp, ws, None) == bsv.VSA_ERR_UNSUPPORTED
        # a wider input row makes the input span larger: an output right after the packed size now overlaps it
        tb = (64 + 64 + 1024) * 2 * 128 * 2
        args = bsv.vsa_forward_args_t(g, 2 * g, 3 * g, 4 * g, g + tb, None, None, 0, 4 * 128)
        assert lib.vsa_forward_ex(plan, ctypes.byref(args), wsp, ws, None) == bsv.VSA_ERR_INVALID_ARG
        assert lib.vsa_forward_lengths(plan, None, ctypes.c_void_p(g), ctypes.c_void_p(2 * g), ctypes.c_void_p(3 * g),
                                       ctypes.c_void_p(4 * g), ctypes.c_void_p(6 * g), wsp, ws,
                                       None) == bsv.VSA_ERR_INVALID_ARG
    finally:
        bsv.vsa_plan_destroy(plan)
        bsv.vsa_plan_destroy(sub)

"""CPU-side checks of the C ABI: the library builds, loads, exports every entry
point include/vdit.h declares, and rejects bad arguments on the host before
touching the GPU."""
import ctypes
import os
import re

import pytest

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "vdit.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return vd.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"VDIT_API\s+[\w\s\*]*?\b(vdit_\w+)\s*\(", text)


def test_header_declares_entry_points():
    names = declared_functions()
    assert set(names) == set(vd.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version(lib):
    assert "sm_103a" in vd.version()


@pytest.mark.parametrize("args,needle", [
    ((4, 48, 1, 0, 15), "multiple of 16"),
    ((4, 48, 1, 0, 0), "multiple of 16"),
    ((4, 50, 1, 0, 16), "does not divide"),
    ((9, 400, 1, 0, 128), "does not divide"),
    ((0, 48, 1, 0, 16), "num_frames"),
    ((4, 0, 1, 0, 16), "tokens_per_frame"),
    ((4, 48, -1, 0, 16), "window_radius"),
    ((4, 48, 1, 4, 16), "ref_frame"),
    ((4, 48, 1, -2, 16), "ref_frame"),
    ((5000, 48, 1, 0, 16), "num_frames"),
    ((2, 1 << 30, 1, 0, 16), "int32"),
])
def test_plan_rejects_bad_arguments(lib, args, needle):
    h = ctypes.c_void_p(1234)
    st = lib.vdit_attn_plan(*args, None, ctypes.byref(h))
    assert st == vd.VDIT_ERR_INVALID
    assert needle in lib.vdit_last_error().decode()
    assert not h.value


def test_plan_null_out(lib):
    assert lib.vdit_attn_plan(4, 48, 1, 0, 16, None, None) == vd.VDIT_ERR_INVALID


def test_key_stats_rejects_bad_arguments(lib):
    s3 = vd._I64x3(8 * 128, 128 * 16, 128)
    p = ctypes.c_void_p(0x1000)
    ws = lib.vdit_key_stats_workspace_size(1, 2, 16, 128)
    assert ws == 2 * 1 * (128 + 2) * 4
    args = [p, p, 1, 2, 16, 128, s3, s3, 0.1, 64.0, p, p, p, p, p, p, ws, None]
    bad = list(args); bad[0] = None
    assert lib.vdit_key_stats(*bad) == vd.VDIT_ERR_INVALID
    bad = list(args); bad[5] = 96
    assert lib.vdit_key_stats(*bad) == vd.VDIT_ERR_UNSUPPORTED
    bad = list(args); bad[16] = ws - 1
    assert lib.vdit_key_stats(*bad) == vd.VDIT_ERR_INVALID
    assert "workspace" in lib.vdit_last_error().decode()
    bad = list(args); bad[0] = ctypes.c_void_p(0x1008)
    assert lib.vdit_key_stats(*bad) == vd.VDIT_ERR_INVALID
    bad = list(args); bad[6] = vd._I64x3(8 * 128, 128 * 16, 100)
    assert lib.vdit_key_stats(*bad) == vd.VDIT_ERR_INVALID
    for scale in (0.0, -0.1, float("inf"), float("nan")):
        bad = list(args); bad[8] = scale
        assert lib.vdit_key_stats(*bad) == vd.VDIT_ERR_INVALID
        assert "scale" in lib.vdit_last_error().decode()
    for tau in (-1.0, float("nan")):
        bad = list(args); bad[9] = tau
        assert lib.vdit_key_stats(*bad) == vd.VDIT_ERR_INVALID


def test_attn_fwd_rejects_null_plan(lib):
    s3 = vd._I64x3(8, 8, 8)
    p = ctypes.c_void_p(0x1000)
    st = lib.vdit_attn_fwd(None, p, p, p, p, 0, None, 1, 1, 128, s3, s3, s3, s3, 0.1, p, p, p, 0, None)
    assert st == vd.VDIT_ERR_INVALID
    assert "plan" in lib.vdit_last_error().decode()


def test_product_path_does_not_import_oracle():
    """The library package never reaches the oracle (no CPU fallback)."""
    pkg = os.path.dirname(vd.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "vdit_oracle" not in text, f


def test_pipeline_entry_points_reject_bad_arguments(lib):
    h = ctypes.c_void_p(1234)
    assert lib.vdit_pipeline_create(None, 1, 8, 128, 2, None, ctypes.byref(h)) == vd.VDIT_ERR_INVALID
    assert "plan" in lib.vdit_last_error().decode()
    assert not h.value
    assert lib.vdit_pipeline_create(ctypes.c_void_p(0x1000), 1, 8, 128, 2, None, None) == vd.VDIT_ERR_INVALID
    sizes = (ctypes.c_int32 * 2)(3, 4)     # sums to 7, not H = 8
    fake_plan = ctypes.c_void_p(0x1000)
    assert lib.vdit_pipeline_create(fake_plan, 1, 8, 128, 2, sizes, ctypes.byref(h)) == vd.VDIT_ERR_INVALID
    assert "sum" in lib.vdit_last_error().decode()
    s3 = vd._I64x3(8, 8, 8)
    p = ctypes.c_void_p(0x1000)
    assert lib.vdit_pipeline_run(None, p, p, p, p, None, s3, 0.1, 64.0, 0, None) == vd.VDIT_ERR_INVALID
    lib.vdit_pipeline_destroy(None)   # NULL is ignored


def test_prologue_entry_points_reject_bad_arguments(lib):
    p = ctypes.c_void_p(0x1000)
    s2 = (ctypes.c_int64 * 2)(1024, 1024)
    s3 = vd._I64x3(8, 8, 8)
    st = lib.vdit_qkv_prologue(None, s2, p, p, p, p, p, s3, s3, s3, 1, 16, 1024, 8, 128, 1e-6, p, 1 << 20, None)
    assert st == vd.VDIT_ERR_INVALID and "NULL" in lib.vdit_last_error().decode()
    st = lib.vdit_qkv_prologue(p, s2, p, p, p, p, p, s3, s3, s3, 1, 16, 1024, 8, 96, 1e-6, p, 1 << 20, None)
    assert st == vd.VDIT_ERR_UNSUPPORTED
    st = lib.vdit_qkv_prologue(p, s2, p, p, p, p, p, s3, s3, s3, 1, 16, 1020, 8, 128, 1e-6, p, 1 << 20, None)
    assert st == vd.VDIT_ERR_INVALID and "multiple of 8" in lib.vdit_last_error().decode()
    st = lib.vdit_qkv_prologue(p, s2, p, p, p, p, p, s3, s3, s3, 1, 16, 1024, 8, 128, 1e-6, p, 16, None)
    assert st == vd.VDIT_ERR_INVALID and "workspace" in lib.vdit_last_error().decode()
    assert lib.vdit_qkv_workspace_size(1, 46800) >= 46800 * 4
    assert lib.vdit_rope_table(None, 16, 128, 1e4, None) == vd.VDIT_ERR_INVALID
    assert lib.vdit_rope_table(p, 16, 127, 1e4, None) == vd.VDIT_ERR_INVALID
    for base in (0.0, float("inf"), float("nan")):
        assert lib.vdit_rope_table(p, 16, 128, base, None) == vd.VDIT_ERR_INVALID
    for eps in (-1e-6, float("inf"), float("nan")):
        st = lib.vdit_qkv_prologue(p, s2, p, p, p, p, p, s3, s3, s3, 1, 16, 1024, 8, 128, eps, p, 1 << 20, None)
        assert st == vd.VDIT_ERR_INVALID and "eps" in lib.vdit_last_error().decode()
    assert lib.vdit_qkv_fold_gamma(None, p, p, 4, 8, None) == vd.VDIT_ERR_INVALID


def test_default_head_groups_cover_every_head(lib):
    """The pipeline's default schedule (host only): the groups cover the H heads
    exactly; from H = 16 (while the groups stay within 64) it ramps 1, 2, 3 up
    and 3, 2, 1 down around middle groups of at least 4 that differ by at most
    one head; otherwise it is an even split into groups of about 4."""
    for H in range(1, 400):
        g = vd.default_groups(H)
        assert sum(g) == H and min(g) >= 1, (H, g)
        mid = g[3:-3]
        if H >= 16 and 6 + (H - 12) // 4 <= 64:   # the ramps fit the 64-group limit
            assert g[:3] == [1, 2, 3] and g[-3:] == [3, 2, 1], (H, g)
            assert min(mid) >= 4 and max(mid) - min(mid) <= 1, (H, g)
        else:
            assert max(g) <= -(-H // -(-H // 4)) and len(g) == -(-H // max(g)), (H, g)
    assert vd.default_groups(24) == [1, 2, 3, 4, 4, 4, 3, 2, 1]
    assert vd.default_groups(19) == [1, 2, 3, 7, 3, 2, 1]
    assert vd.default_groups(8) == [4, 4]
    buf = (ctypes.c_int32 * 2)()
    assert lib.vdit_pipeline_default_groups(24, ctypes.cast(buf, ctypes.c_void_p), 2) == 0
    assert lib.vdit_pipeline_default_groups(0, ctypes.cast(buf, ctypes.c_void_p), 2) == 0


def test_plan_part_rejects_bad_arguments(lib):
    """Plans of one mask part (the two-pass ablation): an unknown part, a mask
    without a reference frame, and a window that covers every frame are refused
    on the host."""
    h = ctypes.c_void_p(1234)
    for args, needle in (((9, 400, 1, 0, 80, 3), "part"), ((9, 400, 1, 0, 80, -1), "part"),
                         ((9, 400, 1, -1, 80, 2), "no reference frame"),
                         ((5, 48, 4, 0, 16, 1), "covers every frame")):
        st = lib.vdit_attn_plan_part(*args, None, ctypes.byref(h))
        assert st == vd.VDIT_ERR_INVALID, args
        assert needle in lib.vdit_last_error().decode(), (args, lib.vdit_last_error())
        assert not h.value


def test_ablation_and_census_entry_points_check_arguments(lib):
    p = ctypes.c_void_p(0x1000)
    s3 = vd._I64x3(8 * 128, 128 * 16, 128)
    assert lib.vdit_plan_block_census(None, 128, p, None) == vd.VDIT_ERR_INVALID
    # two passes need both plans; the workspace size covers fp32 O and LSE of both passes
    args = [None, None, p, p, p, p, 0, None, 1, 2, 128, s3, s3, s3, s3, 0.1, p, p, p, 0, 0, p, 0, None]
    assert lib.vdit_attn_fwd_two_pass(*args) == vd.VDIT_ERR_INVALID
    B, H, N, D = 1, 2, 300, 128
    al = lambda x: (x + 255) // 256 * 256
    assert lib.vdit_attn_two_pass_workspace_size(B, H, N, D) == 2 * (al(B * H * N * D * 4) + al(B * H * N * 4))
    assert lib.vdit_attn_two_pass_workspace_size(0, H, N, D) == 0
    assert lib.vdit_attn_fwd_tiles128(None, p, p, p, p, 0, None, 1, 2, 128, s3, s3, s3, s3, 0.1, p, p, p, 0,
                                      None) == vd.VDIT_ERR_INVALID
    lib.vdit_set_launch_fail_after(0)

"""The allocation-free key-statistics entry point, vdit_key_stats_noalloc.

It serves callers that may not allocate device memory (a plugin whose host
framework owns all device buffers and forbids cudaMalloc, or a loop that cannot
pay cudaMalloc's implicit synchronisation): its scratch is a fixed array inside
the library. These tests call it through the C ABI and compare it with
vdit_key_stats (caller-provided workspace) on two calls in a row with different
inputs and sizes, so state left in the shared array by the first call cannot
leak into the second. Both entry points run the same kernels in the same fixed
reduction order, so their results must be equal bit for bit; each result is also
checked against the fp64 oracle (relative 1e-5, eligibility exact), so a fault
that corrupted both the same way would still fail. This file is collected last
on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import _build, configs, synth

import oracle

pytestmark = pytest.mark.gpu


def _lib():
    _build.build()
    lib = vd.load_library()
    f = lib.vdit_key_stats_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    f.argtypes = [vp, vp, i32, i32, i32, i32, vd._I64x3, vd._I64x3, f32, f32, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return lib


def _outputs(B, H, D):
    return dict(k_mean=torch.full((B, H, D), float("nan"), device="cuda"),
                k_rmax=torch.full((B, H), float("nan"), device="cuda"),
                q_nmax=torch.full((B, H), float("nan"), device="cuda"),
                gap=torch.full((B, H), float("nan"), device="cuda"),
                eligible=torch.full((B, H), 7, dtype=torch.uint8, device="cuda"))


def _noalloc(lib, q, k, scale, tau=64.0):
    B, H, N, D = q.shape
    out = _outputs(B, H, D)
    st = lib.vdit_key_stats_noalloc(
        vd._ptr(q), vd._ptr(k), B, H, N, D, vd._strides(q), vd._strides(k), scale, tau,
        vd._ptr(out["k_mean"]), vd._ptr(out["k_rmax"]), vd._ptr(out["q_nmax"]),
        vd._ptr(out["gap"]), vd._ptr(out["eligible"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == vd.VDIT_OK, lib.vdit_last_error().decode()
    return out


def _compare(got, want):
    """Bitwise equality with the workspace entry point."""
    for key in ("k_mean", "k_rmax", "q_nmax", "gap", "eligible"):
        assert torch.equal(got[key], want[key]), key


def _against_oracle(got, q, k, scale, tau=64.0):
    ref = oracle.key_stats(q.cpu(), k.cpu(), scale, tau)
    c = ref["c"]
    assert np.abs(got["k_mean"].double().cpu().numpy() - c).max() <= 1e-5 * np.abs(c).max() + 1e-6
    for key, rk in (("k_rmax", "R"), ("q_nmax", "qmax"), ("gap", "G")):
        np.testing.assert_allclose(got[key].double().cpu().numpy(), ref[rk], rtol=1e-5, err_msg=key)
    assert np.array_equal(got["eligible"].cpu().numpy(), ref["elig"])


def test_noalloc_matches_workspace_version_two_calls():
    lib = _lib()
    for w in (configs.SMALL, configs.TINY.with_(B=2, H=3, outlier_heads=(0,))):
        q, k, _ = synth.make_qkv(w)
        q, k = q.cuda(), k.cuda()
        got = _noalloc(lib, q, k, w.scale)
        want = vd.key_stats(q, k, w.scale)
        torch.cuda.synchronize()
        _compare(got, want)
        _against_oracle(got, q, k, w.scale)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib()
    # 1 x 64 heads x 2^20 tokens x D=128 needs 64*1024*130*4 bytes > 4 MiB: rejected on
    # the host before any launch, so dummy (aligned, never dereferenced) pointers are fine.
    p = ctypes.c_void_p(1 << 20)
    s3 = vd._I64x3(64 * (1 << 20) * 128, (1 << 20) * 128, 128)
    st = lib.vdit_key_stats_noalloc(p, p, 1, 64, 1 << 20, 128, s3, s3, 0.1, 64.0, p, p, p, p, p,
                                    None)
    assert st == vd.VDIT_ERR_INVALID
    assert "scratch" in lib.vdit_last_error().decode()

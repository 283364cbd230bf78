"""Allocation-failure injection (a host-side test hook, no GPU fault): every
device allocation of plan and pipeline creation is made to fail in turn. Each
failing call must return VDIT_ERR_NOMEM with nothing leaked, and the next
creation must work and give the same schedule."""
import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs

pytestmark = pytest.mark.gpu

PLAN_ALLOCATIONS = 9   # header, frame runs, segments, units, class offsets, gathered tiles, status,
                       # row_ptr, col_idx


def make_plan(w):
    return vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)


def test_every_plan_allocation_failure_is_reported_and_clean():
    w = configs.SMALL
    ref = make_plan(w)
    want = (ref.row_ptr().cpu().numpy(), ref.col_idx().cpu().numpy(), ref.units().cpu().numpy())
    torch.cuda.synchronize()
    try:
        for n in range(1, PLAN_ALLOCATIONS + 1):
            vd.set_alloc_fail_after(n)
            with pytest.raises(vd.VditError) as ei:
                make_plan(w)
            assert ei.value.status == vd.VDIT_ERR_NOMEM, (n, str(ei.value))
            assert "allocation" in str(ei.value)
        # one more allocation than creation makes: the hook is not reached
        vd.set_alloc_fail_after(PLAN_ALLOCATIONS + 1)
        ok = make_plan(w)
        ok.close()
    finally:
        vd.set_alloc_fail_after(0)
    got = make_plan(w)
    assert np.array_equal(got.row_ptr().cpu().numpy(), want[0])
    assert np.array_equal(got.col_idx().cpu().numpy(), want[1])
    assert np.array_equal(got.units().cpu().numpy(), want[2])


def test_failed_creations_leak_nothing():
    """A failure at the last allocation (col_idx) must free the row pointers,
    150 KB for the 1080p-like schedule at block size 16: 100 leaked copies would
    show as 15 MB less free device memory."""
    w = configs.SR1080
    vd.attn_plan(w.F, w.T, w.W, w.ref, 16).close()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    try:
        for _ in range(100):
            vd.set_alloc_fail_after(PLAN_ALLOCATIONS)
            with pytest.raises(vd.VditError):
                vd.attn_plan(w.F, w.T, w.W, w.ref, 16)
    finally:
        vd.set_alloc_fail_after(0)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 < (4 << 20), (free0, free1)


def test_pipeline_allocation_failure():
    w = configs.SMALL
    plan = make_plan(w)
    try:
        vd.set_alloc_fail_after(1)
        with pytest.raises(vd.VditError) as ei:
            vd.Pipeline(plan, w.B, w.H, w.D, 2)
        assert ei.value.status == vd.VDIT_ERR_NOMEM
    finally:
        vd.set_alloc_fail_after(0)
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 2)
    pipe.close()

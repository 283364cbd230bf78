"""Failure detection without a GPU fault: every wait inside the attention kernel
is bounded. With the bound shortened to 1 ns, a normal call must give up early,
drain, free its tensor memory, exit, and report VDIT_ERR_TIMEOUT through the
plan's status word; the context stays usable and the next call, with the
default bound, is correct. The public calls surface the expired wait: attn_fwd
and Pipeline.run raise unless the caller opts out with check=False. A pipeline
run that fails part-way (a refused launch, injected on the host) leaves the
caller's stream waiting for every copy it had queued."""
import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

from parity_util import check_close, oracle_rows

pytestmark = pytest.mark.gpu


def _inputs(w):
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    return (q, k, v), plan


def test_expired_waits_are_reported_and_recoverable():
    w = configs.SMALL
    (q, k, v), plan = _inputs(w)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    st = vd.key_stats(qd, kd, w.scale)
    torch.cuda.synchronize()
    try:
        vd.set_wait_limit_ns(1)
        vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32, check=False)
        torch.cuda.synchronize()
        code = plan.status()
    finally:
        vd.set_wait_limit_ns(0)
    assert code != 0, "a 1 ns bound must expire in at least one wait"
    assert plan.status() == 0, "the status word is cleared once read"
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plan.status() == 0
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, "after timeout")


def test_attn_fwd_raises_on_an_expired_wait_by_default():
    w = configs.SMALL
    (q, k, v), plan = _inputs(w)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    st = vd.key_stats(qd, kd, w.scale)
    torch.cuda.synchronize()
    try:
        vd.set_wait_limit_ns(1)
        with pytest.raises(vd.VditError) as ei:
            vd.attn_fwd(plan, qd, kd, vd_, st, w.scale)
    finally:
        vd.set_wait_limit_ns(0)
    assert ei.value.status == vd.VDIT_ERR_TIMEOUT and "incomplete" in str(ei.value)
    assert plan.status() == 0


def test_pipeline_run_raises_on_an_expired_wait_and_recovers():
    w = configs.SMALL
    (q, k, v), plan = _inputs(w)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    o_h = torch.empty_like(q_h).pin_memory()
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 4)
    torch.cuda.synchronize()
    try:
        vd.set_wait_limit_ns(1)
        with pytest.raises(vd.VditError) as ei:
            pipe.run(q_h, k_h, v_h, o_h, w.scale)
    finally:
        vd.set_wait_limit_ns(0)
    assert ei.value.status == vd.VDIT_ERR_TIMEOUT
    assert plan.status() == 0
    # the next run, with the default bound, is complete and correct
    o_h.zero_()
    pipe.run(q_h, k_h, v_h, o_h, w.scale)
    o_ref, _, _ = oracle_rows(w, q, k, v)
    check_close(o_h.reshape(-1, w.D).double().numpy(), o_ref, what="pipeline after timeout")


def test_pipeline_failing_part_way_joins_the_callers_stream():
    """The third group's attention launch is refused: the run returns
    VDIT_ERR_CUDA after the first two groups (and the third group's copy-in and
    statistics) were queued. Synchronising the caller's stream must then cover
    those copies: the first two groups' outputs are complete, bit for bit those
    of a full run, and the pipeline stays usable."""
    w = configs.SMALL                      # 8 heads, groups of 2
    (q, k, v), plan = _inputs(w)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    want = torch.empty_like(q_h).pin_memory()
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 4)
    pipe.run(q_h, k_h, v_h, want, w.scale)
    o_h = torch.full_like(q_h, float("nan")).pin_memory()
    stream = torch.cuda.current_stream()
    try:
        vd.set_launch_fail_after(3)
        with pytest.raises(vd.VditError) as ei:
            pipe.run(q_h, k_h, v_h, o_h, w.scale, check=False)
    finally:
        vd.set_launch_fail_after(0)
    assert ei.value.status == vd.VDIT_ERR_CUDA and "injected" in str(ei.value)
    stream.synchronize()
    assert torch.equal(o_h[:, :4].view(torch.int16), want[:, :4].view(torch.int16))
    assert torch.isnan(o_h[:, 4:].float()).all(), "groups after the failure were not run"
    assert plan.status() == 0
    o_h.zero_()
    pipe.run(q_h, k_h, v_h, o_h, w.scale)
    assert torch.equal(o_h.view(torch.int16), want.view(torch.int16))

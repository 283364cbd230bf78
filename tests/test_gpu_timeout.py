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


# A bounded wait checks its clock every 32 polls, so a 1 ns bound expires only in a
# wait that needs more polls than that. With the 720p-like geometry (4 heads, about
# five work units per CTA of some 150 key tiles each) the TMA warp waits for the next
# unit's query-tile slot for the whole length of a unit, far beyond 32 polls.
LONG = configs.SR720.with_(name="sr720p_h4", H=4, outlier_heads=(3,))


def test_expired_waits_are_reported_and_recoverable():
    lw = LONG
    (lq, lk, lv), lplan = _inputs(lw)
    lq, lk, lv = lq.cuda(), lk.cuda(), lv.cuda()
    lst = vd.key_stats(lq, lk, lw.scale)
    torch.cuda.synchronize()
    try:
        vd.set_wait_limit_ns(1)
        vd.attn_fwd(lplan, lq, lk, lv, lst, lw.scale, check=False)
        torch.cuda.synchronize()
        code = lplan.status()
    finally:
        vd.set_wait_limit_ns(0)
    assert code != 0, "a 1 ns bound must expire in at least one wait"
    assert lplan.status() == 0, "the status word is cleared once read"
    # the context stays usable: the same plan, then another one, with the default bound
    vd.attn_fwd(lplan, lq, lk, lv, lst, lw.scale)
    w = configs.SMALL
    (q, k, v), plan = _inputs(w)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    st = vd.key_stats(qd, kd, w.scale)
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plan.status() == 0
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, "after timeout")


def test_attn_fwd_raises_on_an_expired_wait_by_default():
    w = LONG
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
    w = LONG
    (q, k, v), plan = _inputs(w)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    o_h = torch.empty_like(q_h).pin_memory()
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 2)
    torch.cuda.synchronize()
    try:
        vd.set_wait_limit_ns(1)
        with pytest.raises(vd.VditError) as ei:
            pipe.run(q_h, k_h, v_h, o_h, w.scale)
    finally:
        vd.set_wait_limit_ns(0)
    assert ei.value.status == vd.VDIT_ERR_TIMEOUT
    assert plan.status() == 0
    # the next run, with the default bound, is complete and equals the single launch
    # bit for bit (grouping by heads leaves every head's arithmetic unchanged)
    o_h.zero_()
    pipe.run(q_h, k_h, v_h, o_h, w.scale)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    want, _ = vd.attn_fwd(plan, qd, kd, vd_, vd.key_stats(qd, kd, w.scale), w.scale, with_lse=False)
    assert torch.equal(o_h.view(torch.int16), want.cpu().view(torch.int16))


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

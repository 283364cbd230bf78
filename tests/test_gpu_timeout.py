"""Failure detection without a GPU fault: every wait inside the attention kernel
is bounded. With the bound shortened to 1 ns, a normal call must give up early,
drain, free its tensor memory, exit, and report VDIT_ERR_TIMEOUT through the
plan's status word; the context stays usable and the next call, with the
default bound, is correct."""
import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

from parity_util import check_close, oracle_rows

pytestmark = pytest.mark.gpu


def test_expired_waits_are_reported_and_recoverable():
    w = configs.SMALL
    q, k, v = synth.make_qkv(w)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    st = vd.key_stats(qd, kd, w.scale)
    torch.cuda.synchronize()
    try:
        vd.set_wait_limit_ns(1)
        vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
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

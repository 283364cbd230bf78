"""Head-group pipelining over host tensors ("Hiding the Collective", Fig. 2):
splitting the heads into groups leaves the token order, and so the mask,
untouched, so the pipelined result must equal the single-launch device path
bit for bit, for any group count and either host layout; one run is also
checked against the fp64 oracle."""
import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

from parity_util import check_close, oracle_rows, stratified_rows

pytestmark = pytest.mark.gpu


def device_reference(w, q, k, v, plan):
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    st = vd.key_stats(qd, kd, w.scale)
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def pinned_like(t):
    return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)


@pytest.mark.parametrize("groups", [1, 3, 8, 0, (1, 2, 5)])
def test_pipeline_equals_single_launch(groups):
    w = configs.SMALL
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    o_ref, lse_ref = device_reference(w, q, k, v, plan)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    o_h = pinned_like(q)
    lse_h = torch.empty((w.B, w.H, w.N), dtype=torch.float32, pin_memory=True)
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, groups)
    pipe.run(q_h, k_h, v_h, o_h, w.scale, lse_h=lse_h)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert torch.equal(o_h.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse_h, lse_ref)
    pipe.close()


@pytest.mark.parametrize("H", [16, 17, 18, 19, 23])
def test_tapered_default_covers_every_head(H):
    """The default schedule (1, 2, 3 heads, groups of 4 with the leftover heads
    spread over them, 3, 2, 1) for head counts whose leftovers outnumber the
    middle groups: every head's output equals the single launch bit for bit."""
    w = configs.Workload(f"taper_h{H}", B=1, H=H, D=64, F=3, T=64, W=1, ref=0, block_size=64,
                         outlier_heads=(H - 1,), seed=40 + H)
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    o_ref, _ = device_reference(w, q, k, v, plan)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    o_h = pinned_like(q)
    o_h.fill_(float("nan"))
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 0)
    pipe.run(q_h, k_h, v_h, o_h, w.scale)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert torch.equal(o_h.view(torch.int16), o_ref.view(torch.int16))
    pipe.close()


def test_pipeline_token_major_host_layout():
    """Host tensors stored [B, N, H, D] (the sequence-sharded layout a projection
    emits) and passed as [B, H, N, D] views: same bytes as the device path."""
    w = configs.SMALL
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    o_ref, _ = device_reference(w, q, k, v, plan)
    tm = [t.permute(0, 2, 1, 3).contiguous().pin_memory().permute(0, 2, 1, 3) for t in (q, k, v)]
    o_store = torch.empty((w.B, w.N, w.H, w.D), dtype=torch.bfloat16, pin_memory=True)
    o_h = o_store.permute(0, 2, 1, 3)
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 3)
    pipe.run(*tm, o_h, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_h.contiguous().view(torch.int16), o_ref.view(torch.int16))


def test_pipeline_matches_oracle_and_repeats():
    """Uneven groups (8 heads in 3 groups), the plan reused across runs, fp64
    oracle on stratified rows (bf16 output: tolerances of the device path)."""
    w = configs.SMALL
    q, k, v = synth.make_qkv(w, seed=11)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 3)
    outs = []
    for _ in range(2):
        o_h = pinned_like(q)
        pipe.run(q_h, k_h, v_h, o_h, w.scale)
        torch.cuda.synchronize()
        outs.append(o_h)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    rows = stratified_rows(w, per_frame_random=4)
    o_ref, _, _ = oracle_rows(w, q, k, v, rows)
    o = outs[0].reshape(-1, w.D)[torch.from_numpy(rows)].double().numpy()
    check_close(o, o_ref, what="pipelined attention")


def test_pipeline_full_size_720p_groups():
    """The 720p-like workload in the library's tapered head groups (1, 2, 3, 4,
    4, 4, 3, 2, 1) equals the single launch."""
    w = configs.SR720
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    o_ref, lse_ref = device_reference(w, q, k, v, plan)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    o_h = pinned_like(q)
    lse_h = torch.empty((w.B, w.H, w.N), dtype=torch.float32, pin_memory=True)
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 0)
    pipe.run(q_h, k_h, v_h, o_h, w.scale, lse_h=lse_h)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert torch.equal(o_h.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse_h, lse_ref)


@pytest.mark.parametrize("w,groups", [(configs.SMALL.with_(name="small_b2", B=2, seed=21), 3),
                                      (configs.TINY, 2)], ids=["b2_d128", "d64"])
def test_pipeline_batches_and_head_dim_64(w, groups):
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    o_ref, lse_ref = device_reference(w, q, k, v, plan)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    o_h = pinned_like(q)
    lse_h = torch.empty((w.B, w.H, w.N), dtype=torch.float32, pin_memory=True)
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, groups)
    pipe.run(q_h, k_h, v_h, o_h, w.scale, lse_h=lse_h)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert torch.equal(o_h.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse_h, lse_ref)


def test_pipeline_rejects_bad_scalars_before_queuing():
    w = configs.TINY
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    o_h = pinned_like(q)
    o_h.fill_(3.0)
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 2)
    for scale in (float("inf"), float("nan"), -1.0):
        with pytest.raises(vd.VditError) as ei:
            pipe.run(q_h, k_h, v_h, o_h, scale)
        assert ei.value.status == vd.VDIT_ERR_INVALID and "scale" in str(ei.value)
    torch.cuda.synchronize()
    assert bool((o_h == 3.0).all()), "a rejected call must not write the output"
    pipe.run(q_h, k_h, v_h, o_h, w.scale)          # the pipeline stays usable
    torch.cuda.synchronize()
    o_ref, _ = device_reference(w, q, k, v, plan)
    assert torch.equal(o_h.view(torch.int16), o_ref.view(torch.int16))
    pipe.close()


def test_pipeline_driven_from_two_streams_in_turn():
    """One pipeline run on stream A and, with no synchronisation in between, again on
    stream B with other host buffers (the 720p-like geometry, 4 heads, groups of one
    head, so the second run's first copies would land in slots the first run's
    kernels still read): a run reuses a device slot only after the previous run's
    kernels and copies of that slot are done, so both outputs equal their single
    launches bit for bit."""
    w = configs.SR720.with_(name="sr720p_h4", H=4, outlier_heads=(3,))
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    ins = [synth.make_qkv(w, seed=s) for s in (5, 6)]
    refs = [device_reference(w, *x, plan)[0] for x in ins]
    hosts = [tuple(t.pin_memory() for t in x) for x in ins]
    outs = [pinned_like(ins[0][0]) for _ in range(2)]
    pipe = vd.Pipeline(plan, w.B, w.H, w.D, 4)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for i in range(2):
        pipe.run(*hosts[i], outs[i], w.scale, stream=streams[i], check=False)
    for s in streams:
        s.synchronize()
    assert plan.status() == 0
    for i in range(2):
        assert torch.equal(outs[i].view(torch.int16), refs[i].view(torch.int16)), i
    pipe.close()

"""GPU parity of the per-segment (windowed) bound: vdit_key_stats_framed against
the oracle's per-query-frame statistics (R, G within relative 1e-5, eligibility
bit-exact), and vdit_attn_fwd_framed against the fp64 oracle rows."""
import numpy as np
import pytest
import torch

import oracle
import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

from parity_util import check_close, gather_rows, oracle_rows, stratified_rows

pytestmark = pytest.mark.gpu

TAU = 64.0
CASES = [
    configs.TINY,
    configs.SMALL,
    configs.Workload("outlier_mid", B=1, H=4, D=128, F=9, T=400, W=1, ref=0, block_size=80,
                     outlier_heads=(2,), seed=21),
    configs.Workload("noref_w0", B=2, H=2, D=128, F=6, T=160, W=0, ref=-1, block_size=32,
                     outlier_heads=(1,), seed=22),
    configs.Workload("dense_small", B=1, H=3, D=64, F=5, T=48, W=4, ref=0, block_size=16,
                     outlier_heads=(2,), seed=23),
    # 16-row tails in gathered tiles: each row takes its own segment's bound, and a
    # tile takes the static path only if every piece's segment is eligible
    configs.Workload("gather_outlier", B=1, H=3, D=128, F=9, T=1040, W=1, ref=0, block_size=80,
                     outlier_heads=(1,), seed=24),
]


def frame_of_segments(plan, w):
    segs = plan.segments().cpu().numpy()
    fmap = np.zeros(w.F, dtype=np.int64)
    for si, s in enumerate(segs):
        fmap[s[0] // w.T:(s[0] + s[1]) // w.T] = si
    return fmap


@pytest.mark.parametrize("w", CASES + [configs.SR720], ids=lambda w: w.name)
def test_framed_stats_parity(w):
    q, k, _ = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    st = vd.key_stats_framed(plan, q.cuda(), k.cuda(), w.scale, TAU)
    torch.cuda.synchronize()
    fs = oracle.frame_stats(q, k, w.T, w.W, w.ref, w.scale, TAU)
    fmap = frame_of_segments(plan, w)
    S = plan.info.n_segments
    # per segment: R is the frame value (frames of one segment see the same keys);
    # Qmax and G take the max over the segment's frames
    Rs = np.zeros((w.B, w.H, S)); Gs = np.zeros((w.B, w.H, S))
    for f in range(w.F):
        Rs[..., fmap[f]] = fs["R"][..., f]
        Gs[..., fmap[f]] = np.maximum(Gs[..., fmap[f]], fs["G"][..., f])
    np.testing.assert_allclose(st["seg_rmax"].double().cpu().numpy(), Rs, rtol=1e-5)
    np.testing.assert_allclose(st["seg_gap"].double().cpu().numpy(), Gs, rtol=1e-5)
    elig_ref = ((Gs.astype(np.float32) <= np.float32(TAU))).astype(np.uint8)
    assert np.array_equal(st["seg_eligible"].cpu().numpy(), elig_ref)
    assert (np.abs(Gs - TAU) > 1e-3 * TAU).all()
    ost = oracle.key_stats(q, k, w.scale, TAU)
    np.testing.assert_allclose(st["k_mean"].double().cpu().numpy(), ost["c"], atol=1e-5 * np.abs(ost["c"]).max() + 1e-6)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_framed_attention_parity(w):
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    st = vd.key_stats_framed(plan, qd, kd, w.scale, TAU)
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plan.status() == 0
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, w.name)


@pytest.mark.parametrize("w", [configs.SR720, configs.SR1080], ids=lambda w: w.name)
def test_framed_full_size_sampled(w):
    q, k, v = synth.make_qkv(w)
    rows = stratified_rows(w, per_frame_random=13 if w is configs.SR720 else 6)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v, rows)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    st = vd.key_stats_framed(plan, qd, kd, w.scale, TAU)
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plan.status() == 0
    check_close(gather_rows(o, rows, w.N), o_ref, gather_rows(lse, rows, w.N), lse_ref, f"{w.name} framed")
    # at least as many eligible (head, segment) pairs as per-head eligibility gives
    head = vd.key_stats(qd, kd, w.scale, TAU)["eligible"].cpu().numpy()
    seg = st["seg_eligible"].cpu().numpy()
    assert (seg >= head[..., None]).all()

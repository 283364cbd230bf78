"""The design before frame alignment, as an ablation ("Deleting the Mask", Fig. 3
of "HeyGen x Google Cloud: Bringing Avatar IV to TPUs"): 128-multiple tiles that
ignore frame boundaries (mask predicates on straddling tiles, sequence padded to
a multiple of 128), and the window and the reference frame run as two passes
merged from fp32 intermediates. Every form must compute the same attention as
the frame-aligned single pass: outputs against the fp64 oracle of the whole
mask (max-abs 1e-2, mean-abs 1e-3 on O, 1e-3 on LSE), all rows on the small
cases and stratified rows at the 720p-like size. The plans of the two mask parts
partition the live pairs: the window part equals the plan without a reference
frame bit for bit, and the reference part holds exactly the reference frame for
the query frames whose window leaves it out."""
import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

import oracle

from parity_util import check_close, gather_rows, oracle_rows, stratified_rows

pytestmark = pytest.mark.gpu

CASES = [
    configs.TINY,                                        # 48-token frames: a 128-row tile spans 3 frames
    configs.SMALL,                                       # 400-token frames (not a multiple of 128)
    configs.Workload("ref_mid", B=2, H=2, D=128, F=7, T=144, W=1, ref=3, block_size=48,
                     outlier_heads=(0,), seed=12),
    configs.Workload("ref_last_d64", B=1, H=3, D=64, F=8, T=208, W=1, ref=7, block_size=16,
                     outlier_heads=(1,), seed=18),
    configs.Workload("w2_t640", B=1, H=2, D=128, F=9, T=640, W=2, ref=0, block_size=128,
                     outlier_heads=(1,), seed=22),   # T a multiple of 128: no partial tile
    # 320 tokens: three 128-row tiles, so the last frame-blind block is a lone tile
    configs.Workload("lone_block", B=2, H=2, D=128, F=4, T=80, W=1, ref=2, block_size=16,
                     outlier_heads=(0,), seed=25),
    # 1040-token frames: the window part's 16-row tails run as gathered tiles
    configs.Workload("gather_parts", B=1, H=2, D=128, F=9, T=1040, W=2, ref=0, block_size=80,
                     outlier_heads=(1,), seed=26),
]


def _dev(w):
    q, k, v = synth.make_qkv(w)
    return (q, k, v), tuple(t.cuda() for t in (q, k, v))


def _plans(w):
    return (vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size, part="window"),
            vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size, part="reference"))


@pytest.mark.parametrize("w", CASES + [configs.DENSE.with_(name="dense_small", F=5, T=104, H=2,
                                                          outlier_heads=(1,), seed=23),
                                       configs.Workload("noref", B=1, H=2, D=128, F=6, T=160, W=0,
                                                        ref=-1, block_size=32, outlier_heads=(1,), seed=11),
                                       # one token, and 40 tokens: a single block, mostly padding
                                       configs.Workload("one_token", B=1, H=2, D=128, F=1, T=1, W=0, ref=0,
                                                        block_size=16, outlier_heads=(), seed=20),
                                       configs.Workload("dense_n40", B=1, H=2, D=64, F=5, T=8, W=4, ref=0,
                                                        block_size=16, outlier_heads=(1,), seed=21)],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("mode", ["auto", "online"])
def test_tiles128_one_pass_all_rows(w, mode):
    (q, k, v), (qd, kd, vd_) = _dev(w)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    st = vd.key_stats(qd, kd, w.scale)
    o, lse = vd.attn_fwd_tiles128(plan, qd, kd, vd_, st, w.scale, mode=mode, out_dtype=torch.float32)
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, f"tiles128 {w.name} {mode}")


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("tiles", ["frame", "128"])
@pytest.mark.parametrize("mode", ["auto", "online"])
def test_two_pass_all_rows(w, tiles, mode):
    (q, k, v), (qd, kd, vd_) = _dev(w)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    pw, pr = _plans(w)
    st = vd.key_stats(qd, kd, w.scale)
    o, lse = vd.attn_fwd_two_pass(pw, pr, qd, kd, vd_, st, w.scale, mode=mode, tiles=tiles,
                                  out_dtype=torch.float32)
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, f"two-pass {tiles} {w.name} {mode}")
    # bf16 output of the merge is the fp32 output rounded to nearest even
    o16, _ = vd.attn_fwd_two_pass(pw, pr, qd, kd, vd_, st, w.scale, mode=mode, tiles=tiles,
                                  out_dtype=torch.bfloat16, with_lse=False)
    torch.cuda.synchronize()
    assert torch.equal(o16, o.to(torch.bfloat16))


@pytest.mark.parametrize("form", ["tiles128", "two_pass_frame", "two_pass_128"])
def test_full_size_720p_sampled_rows(form):
    """The 720p-like workload in each ablation form, as the ablation benchmark
    times it (AUTO mode, one head on the online path)."""
    w = configs.SR720
    (q, k, v), (qd, kd, vd_) = _dev(w)
    rows = stratified_rows(w, per_frame_random=3)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v, rows)
    st = vd.key_stats(qd, kd, w.scale)
    if form == "tiles128":
        plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
        o, lse = vd.attn_fwd_tiles128(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
    else:
        pw, pr = _plans(w)
        o, lse = vd.attn_fwd_two_pass(pw, pr, qd, kd, vd_, st, w.scale, out_dtype=torch.float32,
                                      tiles="frame" if form == "two_pass_frame" else "128")
    check_close(gather_rows(o, rows, w.N), o_ref, gather_rows(lse, rows, w.N), lse_ref, form)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("F,T,W,ref,bs", [(4, 48, 1, 0, 16), (9, 400, 1, 0, 80), (13, 3600, 2, 0, 240),
                                          (7, 144, 1, 3, 48), (8, 48, 1, 7, 16), (9, 8160, 1, 0, 240)])
def test_plan_parts_partition_the_mask(F, T, W, ref, bs):
    full = vd.attn_plan(F, T, W, ref, bs)
    pw = vd.attn_plan(F, T, W, ref, bs, part="window")
    pr = vd.attn_plan(F, T, W, ref, bs, part="reference")
    assert pw.info.part == 1 and pr.info.part == 2 and full.info.part == 0
    assert pw.live_pairs + pr.live_pairs == full.live_pairs
    # the window part is the plan without a reference frame
    want = oracle.schedule(F, T, W, -1, bs)
    assert pw.live_pairs == want.live_pairs
    assert np.array_equal(pw.row_ptr().cpu().numpy(), want.row_ptr)
    assert np.array_equal(pw.col_idx().cpu().numpy(), want.col_idx)
    assert np.array_equal(pw.frame_runs().cpu().numpy(), want.runs)
    # the reference part: frame ref alone, for the frames farther than W from it
    runs = pr.frame_runs().cpu().numpy()
    for f in range(F):
        sees = abs(f - ref) > W
        assert list(runs[f]) == ([ref * T, (ref + 1) * T, 0, 0] if sees else [0, 0, 0, 0])
    n_far = sum(abs(f - ref) > W for f in range(F))
    assert pr.live_pairs == n_far * T * T
    row_ptr, col = pr.row_ptr().cpu().numpy(), pr.col_idx().cpu().numpy()
    per = T // bs
    for qb in range(F * T // bs):
        f = qb // per
        blocks = list(range(ref * per, (ref + 1) * per)) if abs(f - ref) > W else []
        assert list(col[row_ptr[qb]:row_ptr[qb + 1]]) == blocks


def test_reference_pass_alone_under_frame_blind_tiles():
    """The reference part alone with the frame-blind tiling: rows of frames whose
    window leaves the reference frame out attend to that frame only (a plain
    softmax over its keys, in float64 here); the other rows see no key and get
    O = 0 and LSE = -inf."""
    w = configs.Workload("refpass", B=1, H=2, D=128, F=6, T=144, W=1, ref=0, block_size=48,
                         outlier_heads=(1,), seed=24)
    (q, k, v), (qd, kd, vd_) = _dev(w)
    pr = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size, part="reference")
    st = vd.key_stats(qd, kd, w.scale)
    o, lse = vd.attn_fwd_tiles128(pr, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    qq, kk, vv = (t.double().numpy() for t in (q, k, v))
    kr, vr = kk[:, :, w.ref * w.T:(w.ref + 1) * w.T], vv[:, :, w.ref * w.T:(w.ref + 1) * w.T]
    s = np.einsum("bhid,bhjd->bhij", qq, kr) * w.scale
    m = s.max(-1, keepdims=True)
    p = np.exp(s - m)
    want_o = np.einsum("bhij,bhjd->bhid", p, vr) / p.sum(-1, keepdims=True)
    want_l = (m[..., 0] + np.log(p.sum(-1)))
    far = np.abs(np.arange(w.N) // w.T - w.ref) > w.W
    check_close(o[:, :, far].reshape(-1, w.D), want_o[:, :, far].reshape(-1, w.D),
                lse[:, :, far].reshape(-1), want_l[:, :, far].reshape(-1), "reference pass")
    assert (o[:, :, ~far] == 0).all() and np.isneginf(lse[:, :, ~far]).all()


def test_two_pass_rejects_mismatched_plans():
    w = configs.SMALL
    (_, _, _), (qd, kd, vd_) = _dev(w)
    st = vd.key_stats(qd, kd, w.scale)
    pw, pr = _plans(w)
    other = vd.attn_plan(w.F, w.T, w.W + 1, w.ref, w.block_size, part="reference")
    for a, b in ((pr, pw), (pw, other)):
        with pytest.raises(vd.VditError) as ei:
            vd.attn_fwd_two_pass(a, b, qd, kd, vd_, st, w.scale)
        assert ei.value.status == vd.VDIT_ERR_INVALID
    with pytest.raises(vd.VditError):
        vd.attn_plan(5, 48, 4, 0, 16, part="window")          # dense: no separate reference part
    with pytest.raises(vd.VditError):
        vd.attn_plan(5, 48, 1, -1, 16, part="reference")      # no reference frame

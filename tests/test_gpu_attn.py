"""GPU parity of the fused attention against the fp64 oracle.

Full-row comparisons on cases the oracle finishes in seconds (several query and
key tiles, ragged key tails, segments shorter than a tile, dense with a key
count that is not a multiple of 16, no reference frame, reference frame in the
middle or last, 16-token frames, a single token, D = 64 and 128, batch > 1,
strided inputs); stratified row samples at the full 720p-like, 1080p-like and
dense sizes, and the 720p-like geometry at D = 64, in the launch configuration
the benchmark times. Tolerances: max-abs 1e-2, mean-abs 1e-3 on O (fp32
output), 1e-3 on LSE; the bf16 output equals the fp32 output rounded to nearest
even.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

import oracle

from parity_util import check_close, gather_rows, oracle_rows, stratified_rows

pytestmark = pytest.mark.gpu

SMALL_CASES = [
    configs.TINY,
    configs.SMALL,
    configs.SMALL.with_(name="small_bs16", block_size=16),
    configs.TINY.with_(name="tiny_d128", D=128, H=3, outlier_heads=(2,)),
    configs.Workload("noref_w0", B=1, H=2, D=128, F=6, T=160, W=0, ref=-1, block_size=32,
                     outlier_heads=(1,), seed=11),
    configs.Workload("ref_mid", B=2, H=2, D=128, F=7, T=144, W=1, ref=3, block_size=48,
                     outlier_heads=(0,), seed=12),
    configs.Workload("dense_tail8", B=1, H=2, D=128, F=21, T=104, W=20, ref=0, block_size=16,
                     outlier_heads=(1,), seed=13),
    configs.Workload("dense_tiny", B=1, H=2, D=64, F=5, T=24, W=4, ref=0, block_size=16,
                     outlier_heads=(), seed=14),
    configs.Workload("one_frame", B=1, H=2, D=128, F=1, T=400, W=0, ref=0, block_size=16,
                     outlier_heads=(1,), seed=15),
    configs.Workload("wide_w", B=1, H=2, D=64, F=10, T=64, W=3, ref=0, block_size=64,
                     outlier_heads=(1,), seed=16),
    configs.SMALL.with_(name="small_d64", D=64, seed=17),
    configs.Workload("ref_last", B=1, H=2, D=128, F=8, T=48, W=1, ref=7, block_size=16,
                     outlier_heads=(1,), seed=18),
    configs.Workload("short_frames_ref_mid", B=1, H=3, D=64, F=7, T=16, W=2, ref=3, block_size=16,
                     outlier_heads=(2,), seed=19),
    # one token (the output is that token's value row) and a 40-token dense sequence
    configs.Workload("one_token", B=1, H=2, D=128, F=1, T=1, W=0, ref=0, block_size=16,
                     outlier_heads=(), seed=20),
    configs.Workload("dense_n40", B=1, H=2, D=64, F=5, T=8, W=4, ref=0, block_size=16,
                     outlier_heads=(1,), seed=21),
] + [
    # frames of 8 whole tiles and a 16-, 48- or 64-row tail: the tails run as gathered
    # tiles (eight, two and two to a tile) in the chained second launch
    configs.Workload("gather_16", B=1, H=2, D=128, F=9, T=1040, W=1, ref=0, block_size=80,
                     outlier_heads=(1,), seed=26),
    configs.Workload("gather_48_d64", B=1, H=2, D=64, F=6, T=1072, W=2, ref=5, block_size=16,
                     outlier_heads=(0,), seed=27),
    configs.Workload("gather_64_noref", B=2, H=1, D=128, F=5, T=1088, W=1, ref=-1, block_size=64,
                     outlier_heads=(), seed=28),
]
GATHER_CASES = SMALL_CASES[-3:]


def run_gpu(w, q, k, v, mode="auto", out_dtype=torch.float32, stats=None):
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    if stats is None:
        stats = vd.key_stats(qd, kd, w.scale)
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, stats, w.scale, mode=mode, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert plan.status() == 0
    return o, lse, stats, plan


@pytest.mark.parametrize("w", SMALL_CASES, ids=lambda w: w.name)
def test_attention_full_rows(w):
    q, k, v = synth.make_qkv(w)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    o, lse, st, _ = run_gpu(w, q, k, v)
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, w.name)
    # the outlier heads are the ineligible ones (they took the online branch)
    elig = st["eligible"].cpu().numpy()
    for h in range(w.H):
        assert elig[:, h].all() == (h not in w.outlier_heads)


@pytest.mark.parametrize("w", SMALL_CASES[:3] + SMALL_CASES[5:7] + GATHER_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("mode", ["online", "static"])
def test_forced_modes_agree(w, mode):
    """FORCE_ONLINE everywhere and FORCE_STATIC on eligible heads match the oracle."""
    q, k, v = synth.make_qkv(w)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    o, lse, st, _ = run_gpu(w, q, k, v, mode=mode)
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    o_ref = o_ref.reshape(o.shape)
    lse_ref = lse_ref.reshape(lse.shape)
    heads = range(w.H) if mode == "online" else [h for h in range(w.H) if h not in w.outlier_heads]
    for h in heads:
        check_close(o[:, h], o_ref[:, h], lse[:, h], lse_ref[:, h], f"{w.name} {mode} h{h}")


def test_bf16_output_is_rounded_fp32_output():
    w = configs.SMALL
    q, k, v = synth.make_qkv(w)
    o32, _, st, plan = run_gpu(w, q, k, v, out_dtype=torch.float32)
    o16, _ = vd.attn_fwd(plan, q.cuda(), k.cuda(), v.cuda(), st, w.scale, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_deterministic_bytes():
    """Two identical calls write identical bytes. The pages' first quality gate
    compares output hashes byte for byte for changes that keep the reduction
    order ("Proving the Pixels Didn't Change")."""
    w = configs.SMALL
    q, k, v = synth.make_qkv(w)
    o1, l1, st, plan = run_gpu(w, q, k, v, out_dtype=torch.bfloat16)
    o2, l2 = vd.attn_fwd(plan, q.cuda(), k.cuda(), v.cuda(), st, w.scale, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_strided_inputs_and_outputs():
    """[B, N, H, D] storage viewed as [B, H, N, D] for Q, K, V and O."""
    w = configs.SMALL.with_(B=2, H=4, outlier_heads=(3,))
    q, k, v = synth.make_qkv(w)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    perm = lambda t: t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    qd, kd, vd_ = perm(q), perm(k), perm(v)
    out = torch.empty((w.B, w.N, w.H, w.D), dtype=torch.float32, device="cuda").permute(0, 2, 1, 3)
    st = vd.key_stats(qd, kd, w.scale)
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out=out)
    torch.cuda.synchronize()
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, "strided")


def test_lse_optional():
    w = configs.TINY
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    st = vd.key_stats(q.cuda(), k.cuda(), w.scale)
    o, lse = vd.attn_fwd(plan, q.cuda(), k.cuda(), v.cuda(), st, w.scale, with_lse=False,
                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lse is None
    o_ref, _, _ = oracle_rows(w, q, k, v)
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref, what="no-lse")


@pytest.mark.parametrize("w", [configs.SR720, configs.SR1080, configs.DENSE, configs.SR720_D64],
                         ids=lambda w: w.name)
def test_full_size_sampled_rows(w):
    """Full-size workloads in the benchmark's launch configuration (AUTO mode,
    bf16 output as timed, fp32 output for the gate), on stratified row samples."""
    q, k, v = synth.make_qkv(w)
    rows = stratified_rows(w)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v, rows)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    st = vd.key_stats(qd, kd, w.scale)
    o32, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
    o16, _ = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.bfloat16, with_lse=False)
    torch.cuda.synchronize()
    assert plan.status() == 0
    check_close(gather_rows(o32, rows, w.N), o_ref, gather_rows(lse, rows, w.N), lse_ref, w.name)
    assert torch.equal(o16, o32.to(torch.bfloat16))
    # properties that hold at any size: every row finite; LSE finite
    assert torch.isfinite(o32).all() and torch.isfinite(lse).all()


def test_gathered_tiles_across_many_frames():
    """512 frames of 1040 tokens, two heads (64 gathered tiles per head, 4096 tile
    pairs): every tail row and the edges of 52 frames (the first two, the last two
    and 48 seeded ones) against the oracle, in AUTO (head 1 online) and with the
    per-segment bound."""
    w = configs.Workload("gather_512", B=1, H=2, D=128, F=512, T=1040, W=2, ref=0, block_size=1040,
                         outlier_heads=(1,), seed=29)
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    assert plan.info.n_gathers == 64 and plan.info.n_units == 4 * w.F
    rng = np.random.default_rng(29)
    frames = sorted(set([0, 1, w.F - 2, w.F - 1] + [int(x) for x in rng.choice(w.F, 48, replace=False)]))
    rows = np.array([bh * w.N + f * w.T + i for bh in range(w.B * w.H) for f in frames
                     for i in [0, 1023] + list(range(1024, w.T))], dtype=np.int64)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v, rows)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    for st in (vd.key_stats(qd, kd, w.scale), vd.key_stats_framed(plan, qd, kd, w.scale)):
        o, lse = vd.attn_fwd(plan, qd, kd, vd_, st, w.scale, out_dtype=torch.float32)
        torch.cuda.synchronize()
        check_close(gather_rows(o, rows, w.N), o_ref, gather_rows(lse, rows, w.N), lse_ref,
                    what="gather_512")


@pytest.mark.parametrize("w", [
    # dense, 65 tiles (the last owns 108 rows): tiles 50-64 become tail tiles
    configs.Workload("tail_dense", B=1, H=2, D=128, F=5, T=1660, W=4, ref=0, block_size=16,
                     outlier_heads=(1,), seed=31),
    # 1080p-like frames: frame 0 (the shortest units) hands its tiles 48-63 over
    configs.Workload("tail_sparse", B=1, H=2, D=128, F=4, T=8160, W=1, ref=0, block_size=240,
                     outlier_heads=(0,), seed=32),
], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", ["auto", "online"])
def test_tail_tiles(w, mode):
    """Plans without gathered tiles and with at least 32 tile pairs per head run the
    tiles of their last 8 pairs as one-tile records in the second launch: every
    row of those tiles, and stratified rows elsewhere, against the oracle."""
    q, k, v = synth.make_qkv(w)
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    gat = plan.gathers().cpu().numpy()
    assert len(gat) in (15, 16) and (gat[:, 0] == 1).all()
    tail_rows = [bh * w.N + i for bh in range(w.B * w.H) for g in gat for i in range(g[9], g[9] + g[10])]
    rows = np.unique(np.concatenate([np.array(tail_rows, dtype=np.int64), stratified_rows(w, per_frame_random=4)]))
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v, rows)
    qd, kd, vd_ = q.cuda(), k.cuda(), v.cuda()
    o, lse = vd.attn_fwd(plan, qd, kd, vd_, vd.key_stats(qd, kd, w.scale), w.scale, mode=mode,
                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_close(gather_rows(o, rows, w.N), o_ref, gather_rows(lse, rows, w.N), lse_ref, what=w.name)


def test_non_finite_scale_is_rejected():
    w = configs.TINY
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    st = vd.key_stats(q, k, w.scale)
    for scale in (float("inf"), float("nan"), 0.0):
        with pytest.raises(vd.VditError) as ei:
            vd.attn_fwd(plan, q, k, v, st, scale)
        assert ei.value.status == vd.VDIT_ERR_INVALID and "scale" in str(ei.value)


def _full_size_check(w, mode, per_frame_random):
    q, k, v = synth.make_qkv(w)
    rows = stratified_rows(w, per_frame_random=per_frame_random)
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v, rows)
    o32, lse, st, plan = run_gpu(w, q, k, v, mode=mode)
    check_close(gather_rows(o32, rows, w.N), o_ref, gather_rows(lse, rows, w.N), lse_ref,
                f"{w.name} {mode}")
    assert torch.isfinite(o32).all() and torch.isfinite(lse).all()
    return st


def test_full_size_forced_online_720p():
    """The online-softmax path (running max, lazy rescale of O) over the 720p-like
    workload's ~150 key tiles per unit, on every head."""
    _full_size_check(configs.SR720, "online", per_frame_random=4)


@pytest.mark.parametrize("w", configs.dense_sweep(), ids=lambda w: w.name)
def test_full_size_dense_sweep(w):
    """Every point of the dense base-DiT eligibility sweep (key offset scale s in
    {0, 0.5, 2} x 0, 1 or 6 of 24 outlier heads) at full size, AUTO mode as
    timed: attention on a light stratified row sample over a key count that is
    not a multiple of 16, and exactly the outlier heads on the online path
    (centring keeps every regular head eligible at every offset scale; at s = 2
    the mean term q.c of the bound is large)."""
    st = _full_size_check(w, "auto", per_frame_random=2)
    elig = st["eligible"].cpu().numpy().reshape(-1)
    want = np.array([0 if h in w.outlier_heads else 1 for h in range(w.H)], dtype=elig.dtype)
    assert np.array_equal(elig, want), (w.name, elig)


def test_batch_of_two_at_720p_geometry():
    """B = 2 with the 720p-like frame geometry (13 x 3600 tokens, window +-2,
    reference frame 0), 2 heads each, one of them an outlier: the batch index
    of every unit, stride and output row at full sequence length."""
    w = configs.SR720.with_(name="sr720p_b2h2", B=2, H=2, outlier_heads=(1,), seed=18)
    _full_size_check(w, "auto", per_frame_random=6)


def _worst_case_gap_inputs(s_heads, R=16.0, T=128, F=4, D=128, seed=31):
    """Block-diagonal mask (W = 0, no reference frame). In every head the keys of
    frame 0 sit at c - R e0 and the keys of frames 1..3 at c + (R/3) e0, so the
    key mean is c and the largest centred key norm is R. Every query of the head
    is s e0. A query in frame 0 sees only the keys of frame 0, so its true max
    logit is scale (q.c - s R) while its bound is scale (q.c + s R): the gap is
    2 scale s R = G, the worst case the eligibility rule allows for."""
    g = torch.Generator().manual_seed(seed)
    H = len(s_heads)
    c = torch.zeros(D, dtype=torch.float64)
    c[1:4] = torch.tensor([0.5, -0.25, 0.125], dtype=torch.float64)
    q = torch.zeros((1, H, F * T, D), dtype=torch.float64)
    k = c.expand(1, H, F * T, D).clone()
    for h, s in enumerate(s_heads):
        q[0, h, :, 0] = s
        k[0, h, :T, 0] -= R
        k[0, h, T:, 0] += R / 3
    v = torch.randn((1, H, F * T, D), generator=g, dtype=torch.float64)
    w = configs.Workload("worst_gap", B=1, H=H, D=D, F=F, T=T, W=0, ref=-1, block_size=16,
                         outlier_heads=(), seed=seed)
    return w, (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16))


def test_static_path_at_the_worst_case_gap():
    """'Unchaining the Softmax' eligibility: with G = 2 scale Qmax R <= 64 no row's
    exponentials can underflow, even when a row's true max sits the full G below
    its bound. Head 0 is built at G = 60 with that worst-case gap on every row of
    frame 0 (the static path must match the oracle); head 1 at G = 150 is
    ineligible and must take the online path."""
    w, (q, k, v) = _worst_case_gap_inputs([21.25, 53.0])
    ost = oracle.key_stats(q, k, w.scale, 64.0)
    G = ost["G"].reshape(-1)
    assert 59.0 < G[0] < 61.0 and G[1] > 140.0
    o_ref, lse_ref, mx = oracle_rows(w, q, k, v)
    m = oracle.row_bounds(q, ost["c"], ost["R"], w.scale).reshape(-1)
    gap0 = (m - mx)[: w.T]                                  # head 0, frame 0 rows
    assert np.allclose(gap0, G[0], rtol=1e-6), "the construction must reach the worst case"
    for mode in ("auto", "static", "online"):
        if mode == "static":
            # forcing the bound is only claimed for eligible heads: check head 0 only
            o, lse, st, _ = run_gpu(w.with_(H=1), q[:, :1].contiguous(), k[:, :1].contiguous(),
                                    v[:, :1].contiguous(), mode=mode)
            n = w.N
            check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref[:n],
                        lse.reshape(-1).double().cpu().numpy(), lse_ref[:n], f"worst gap {mode}")
            continue
        o, lse, st, _ = run_gpu(w, q, k, v, mode=mode)
        check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                    lse.reshape(-1).double().cpu().numpy(), lse_ref, f"worst gap {mode}")
        assert st["eligible"].cpu().numpy().reshape(-1).tolist() == [1, 0]


@pytest.mark.parametrize("zero", ["k", "q"])
def test_degenerate_zero_keys_or_queries(zero):
    """All keys zero (c = 0, R = 0, G = 0: eligible, and the bound equals the true
    max 0) or all queries zero (every logit 0): every p is 1, so O is the plain
    mean of V over the row's live keys and LSE = ln |J(i)|. Expected values from
    the frame-window rule directly."""
    w = configs.Workload("zero_" + zero, B=1, H=2, D=128, F=6, T=48, W=1, ref=0, block_size=16,
                         outlier_heads=(), seed=41)
    q, k, v = synth.make_qkv(w)
    if zero == "k":
        k = torch.zeros_like(k)
    else:
        q = torch.zeros_like(q)
    o, lse, st, _ = run_gpu(w, q, k, v)
    assert st["eligible"].cpu().numpy().all()
    vv = v.double().numpy()[0]                          # [H, N, D]
    f = np.arange(w.N) // w.T
    live = (np.abs(f[:, None] - f[None, :]) <= w.W) | (f[None, :] == w.ref)   # [N, N]
    want = np.einsum("ij,hjd->hid", live.astype(np.float64), vv) / live.sum(1)[None, :, None]
    got = o[0].double().cpu().numpy()
    assert np.abs(got - want).max() < 1e-5, np.abs(got - want).max()
    np.testing.assert_allclose(lse[0].double().cpu().numpy(),
                               np.broadcast_to(np.log(live.sum(1)), (w.H, w.N)), atol=1e-5)


def test_online_rescale_under_a_rising_max():
    """Online softmax with the row max rising on every key tile (FORCE_ONLINE, one
    1536-token frame = 12 key tiles). Head 0: logits climb ~150 nats along the keys,
    so each tile lifts the running max past the lazy-rescale threshold (2^8) and O
    is rescaled every tile. Head 1: the climb is 60 nats, so some tiles stay under the
    threshold and their p run above 1 against a stale max. Head 2: the logits fall,
    so the first tile holds the max. All rows against the oracle."""
    T, D = 1536, 128
    w = configs.Workload("rising_max", B=1, H=3, D=D, F=1, T=T, W=0, ref=0, block_size=16,
                         outlier_heads=(), seed=43)
    g = torch.Generator().manual_seed(43)
    s = 8.0                                          # |q| along e0
    ramp = torch.arange(T, dtype=torch.float64) / T
    q = torch.zeros((1, 3, T, D), dtype=torch.float64)
    q[..., 0] = s
    q[..., 1:] = 0.05 * torch.randn((1, 3, T, D - 1), generator=g, dtype=torch.float64)
    k = 0.05 * torch.randn((1, 3, T, D), generator=g, dtype=torch.float64)
    for h, total_nats in enumerate((150.0, 60.0, -150.0)):
        k[0, h, :, 0] += total_nats / (w.scale * s) * ramp
    v = torch.randn((1, 3, T, D), generator=g, dtype=torch.float64)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    o_ref, lse_ref, _ = oracle_rows(w, q, k, v)
    o, lse, _, _ = run_gpu(w, q, k, v, mode="online")
    check_close(o.reshape(-1, w.D).double().cpu().numpy(), o_ref,
                lse.reshape(-1).double().cpu().numpy(), lse_ref, "rising max")

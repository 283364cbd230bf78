"""GPU parity of the fused pre-attention chain ("Layout Is the ABI", Fig. 5):
RMSNorm -> q/k/v projection -> rotary embedding -> [B, H, N, D], against the
fp64 oracle, through the C ABI.

Tolerance, derived from the arithmetic of the GPU path:
  * the output is rounded once to bf16 (8 significant bits): |err| <= 2^-8 |z|;
  * everything before it is fp32 (accumulation of bf16 products, 1/rms, the
    rotation): relative error near 1e-6, covered by a 1% margin on the bound
    above and an absolute floor of 2^-16 rms(z);
  * the RMSNorm gain is folded into the weights and rounded to bf16 once. With
    gains that are powers of two (``exact_gain``) that rounding is exact and
    the bound above is the whole tolerance; with general gains each weight
    carries a relative error <= 2^-8, so z_o gains at most 2^-8 sum_c |y_c w_oc|
    (and a rotated element the sum over its pair), checked per element, with
    the statistical check rms(err) <= 2^-7 rms(z)."""
import numpy as np
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

import oracle

pytestmark = pytest.mark.gpu

U8 = 2.0 ** -8


def sample_rows(s, n_random=40, seed=7):
    """Flattened token rows b*N + n: tile edges, the ragged tail, seeded random."""
    rng = np.random.default_rng(seed)
    picks = set()
    for b in range(s.B):
        base = b * s.N
        for n in (0, 1, 127, 128, 129, s.N - 129, s.N - 128, s.N - 2, s.N - 1,
                  (s.N // 128) * 128, (s.N // 128) * 128 - 1):
            if 0 <= n < s.N:
                picks.add(base + n)
        picks.update(int(base + r) for r in rng.integers(0, s.N, n_random))
    return np.array(sorted(picks), dtype=np.int64)


def run_gpu(s, x, w, gamma, out=None, stream=None):
    xd, wd = x.cuda(), w.cuda()
    wf = vd.fold_gamma(wd, gamma.cuda())
    cs = vd.rope_table(s.N, s.D, s.base)
    return vd.qkv_prologue(xd, wf, cs, s.H, s.D, s.eps, out=out)


def gpu_rows(t, rows, N):
    """[B, H, N, D] CUDA tensor -> float64 [len(rows), H, D] for flat rows b*N + n."""
    B, H, _, D = t.shape
    b = torch.from_numpy(rows // N).to(t.device)
    n = torch.from_numpy(rows % N).to(t.device)
    return t[b, :, n, :].double().cpu().numpy()


def abs_sums(s, x, w, gamma, rows):
    """sum_c |y_c w_oc| for the sampled rows, y the normalised, gained hidden row."""
    xr = x.reshape(-1, s.C)[torch.from_numpy(rows)].double().numpy()
    y = xr / np.sqrt((xr ** 2).mean(-1, keepdims=True) + s.eps) * gamma.double().numpy()
    return np.abs(y) @ np.abs(w.double().numpy()).T            # [rows, O]


def check(s, got, ref, rows, sums=None):
    worst = 0.0
    for part, (g, r) in enumerate(zip(got, ref)):
        g = gpu_rows(g, rows, s.N)
        err = np.abs(g - r)
        floor = 2.0 ** -16 * np.sqrt((r ** 2).mean())
        tol = 1.01 * U8 * np.abs(r) + floor
        if sums is not None:
            S = sums[:, part * s.H * s.D:(part + 1) * s.H * s.D].reshape(len(rows), s.H, s.D)
            if part < 2:      # a rotated element mixes the pair (i, i + D/2)
                S = S + np.concatenate([S[..., s.D // 2:], S[..., : s.D // 2]], axis=-1)
            tol = tol + 1.01 * U8 * S
            rel = np.sqrt((err ** 2).mean() / (r ** 2).mean())
            assert rel <= 2.0 ** -7, f"{s.name} part {'qkv'[part]}: rms error {rel:.2e} of rms"
        bad = err > tol
        assert not bad.any(), (f"{s.name} part {'qkv'[part]}: {bad.sum()} elements out of tolerance, "
                               f"worst {(err - tol).max():.3e} over")
        worst = max(worst, float((err / np.maximum(tol, 1e-30)).max()))
    return worst


def test_fold_gamma_bit_exact_and_in_place():
    torch.manual_seed(0)
    w = (torch.randn(384, 200) * 0.1).to(torch.bfloat16)
    g = 1.0 + 0.3 * torch.randn(200)
    want = (w.float() * g).to(torch.bfloat16)
    got = vd.fold_gamma(w.cuda(), g.cuda()).cpu()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    wd = w.cuda()
    vd.fold_gamma(wd, g.cuda(), out=wd)
    assert torch.equal(wd.cpu().view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("N,D,base", [(200, 64, 10000.0), (46800, 128, 10000.0), (77, 128, 500.0)])
def test_rope_table_matches_fp64(N, D, base):
    t = vd.rope_table(N, D, base).cpu().double().numpy()
    i = np.arange(D // 2)[:, None]
    n = np.arange(N)[None, :]
    a = n * base ** (-2.0 * i / D)
    np.testing.assert_allclose(t[..., 0], np.cos(a).astype(np.float32), rtol=0, atol=1.2e-7)
    np.testing.assert_allclose(t[..., 1], np.sin(a).astype(np.float32), rtol=0, atol=1.2e-7)


@pytest.mark.parametrize("s", [configs.PRO_TINY, configs.PRO_RAGGED], ids=lambda s: s.name)
def test_prologue_all_rows_exact_gain(s):
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed, exact_gain=True)
    got = run_gpu(s, x, w, gamma)
    torch.cuda.synchronize()
    rows = np.arange(s.B * s.N, dtype=np.int64)
    ref = oracle.qkv_prologue(x, w, gamma.double().numpy(), s.H, s.D, s.eps, s.base, rows)
    check(s, got, ref, rows)


def test_prologue_column_bands_all_rows():
    """A projection large enough that the GEMM walks its output columns in two
    bands (one per 24 MB of W'), with an uneven last band and a half-wide last
    column tile: every row against the oracle."""
    s = configs.PRO_BANDS
    assert -(-s.O * s.C * 2 // (24 << 20)) == 2      # the band rule of the library
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed, exact_gain=True)
    got = run_gpu(s, x, w, gamma)
    torch.cuda.synchronize()
    rows = np.arange(s.B * s.N, dtype=np.int64)
    ref = oracle.qkv_prologue(x, w, gamma.double().numpy(), s.H, s.D, s.eps, s.base, rows)
    check(s, got, ref, rows)


def test_prologue_general_gain():
    s = configs.PRO_RAGGED
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed + 10)
    got = run_gpu(s, x, w, gamma)
    torch.cuda.synchronize()
    rows = np.arange(s.B * s.N, dtype=np.int64)
    ref = oracle.qkv_prologue(x, w, gamma.double().numpy(), s.H, s.D, s.eps, s.base, rows)
    check(s, got, ref, rows, sums=abs_sums(s, x, w, gamma, rows))


@pytest.mark.parametrize("s", [configs.PRO_SMALL, configs.PRO_SR720], ids=lambda s: s.name)
def test_prologue_sampled_rows(s):
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed, exact_gain=True)
    got = run_gpu(s, x, w, gamma)
    torch.cuda.synchronize()
    rows = sample_rows(s)
    ref = oracle.qkv_prologue(x, w, gamma.double().numpy(), s.H, s.D, s.eps, s.base, rows)
    check(s, got, ref, rows)


def test_prologue_strided_io_and_padding_untouched():
    """x with a padded row stride; q, k, v written into views of one packed
    buffer with padded token rows: the padding keeps its sentinel."""
    s = configs.PRO_RAGGED
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed, exact_gain=True)
    xpad = torch.zeros((s.B, s.N, s.C + 24), dtype=torch.bfloat16)
    xpad[..., : s.C] = x
    xv = xpad.cuda()[..., : s.C]
    sentinel = -7.0
    packed = torch.full((3, s.B, s.H, s.N, s.D + 64), sentinel, dtype=torch.bfloat16, device="cuda")
    outs = tuple(packed[i, ..., : s.D] for i in range(3))
    wf = vd.fold_gamma(w.cuda(), gamma.cuda())
    cs = vd.rope_table(s.N, s.D, s.base)
    vd.qkv_prologue(xv, wf, cs, s.H, s.D, s.eps, out=outs)
    torch.cuda.synchronize()
    assert bool((packed[..., s.D:] == sentinel).all())
    rows = np.arange(s.B * s.N, dtype=np.int64)
    ref = oracle.qkv_prologue(x, w, gamma.double().numpy(), s.H, s.D, s.eps, s.base, rows)
    check(s, outs, ref, rows)


def test_prologue_deterministic():
    s = configs.PRO_SMALL
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed)
    a = [t.clone() for t in run_gpu(s, x, w, gamma)]
    b = run_gpu(s, x, w, gamma)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


def test_prologue_output_feeds_attention():
    """The prologue's [B, H, N, D] outputs are attention's inputs as they are:
    GPU chain (prologue -> key statistics -> attention) against the oracle chain
    (fp64 prologue, rounded to bf16 -> fp64 attention), attention tolerances."""
    from parity_util import check_close, gather_rows, stratified_rows
    wl = configs.SMALL
    s = configs.PrologueShape("chain_small", B=1, N=wl.N, C=wl.H * wl.D, H=wl.H, D=wl.D, seed=5)
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed)
    q, k, v = run_gpu(s, x, w, gamma)
    plan = vd.attn_plan(wl.F, wl.T, wl.W, wl.ref, wl.block_size)
    st = vd.key_stats(q, k, wl.scale)
    o, _ = vd.attn_fwd(plan, q, k, v, st, wl.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.qkv_prologue(x, w, gamma.double().numpy(), s.H, s.D, s.eps, s.base)
    to_bhnd = lambda a: torch.from_numpy(a.reshape(s.B, s.N, s.H, s.D)).permute(0, 2, 1, 3) \
        .contiguous().to(torch.bfloat16)
    rows = stratified_rows(wl, per_frame_random=4)
    o_ref, _, _ = oracle.attention_rows(to_bhnd(rq), to_bhnd(rk), to_bhnd(rv), wl.T, wl.W, wl.ref,
                                        wl.scale, rows)
    check_close(gather_rows(o, rows, wl.N), o_ref, what="prologue -> attention")


def test_prologue_expired_wait_is_reported_and_recoverable():
    s = configs.PRO_SMALL
    x, w, gamma = synth.make_prologue_inputs(s.B, s.N, s.C, s.H, s.D, s.seed, exact_gain=True)
    xd, wf = x.cuda(), vd.fold_gamma(w.cuda(), gamma.cuda())
    cs = vd.rope_table(s.N, s.D, s.base)
    ws = torch.zeros(vd.qkv_workspace_bytes(s.B, s.N), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    try:
        vd.set_wait_limit_ns(1)
        vd.qkv_prologue(xd, wf, cs, s.H, s.D, s.eps, workspace=ws)
        code = vd.qkv_status(ws)
    finally:
        vd.set_wait_limit_ns(0)
    assert code != 0, "a 1 ns bound must expire in at least one wait"
    assert vd.qkv_status(ws) == 0, "the status word is cleared once read"
    got = vd.qkv_prologue(xd, wf, cs, s.H, s.D, s.eps, workspace=ws)
    assert vd.qkv_status(ws) == 0
    rows = sample_rows(s, n_random=16)
    ref = oracle.qkv_prologue(x, w, gamma.double().numpy(), s.H, s.D, s.eps, s.base, rows)
    check(s, got, ref, rows)

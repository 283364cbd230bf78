"""Pins for the oracle's masked attention, row bound and key statistics.

Sources ("HeyGen x Google Cloud: Bringing Avatar IV to TPUs"):
  "Deleting the Mask"      -- window + reference-frame mask, one softmax over it
  "Unchaining the Softmax" -- Cauchy-Schwarz row bound from the key mean and the
                              largest centred key norm; centring leaves the
                              softmax unchanged in exact arithmetic; the bound
                              holds for every row's slice of keys.
The oracle is checked against torch's float64 scaled_dot_product_attention
(dense, block-diagonal and Kronecker-masked cases), scipy's logsumexp, numpy's
mean/norm, invariances and closed forms -- never against itself.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from block_sparse_video_frame_gb300 import configs, synth


def rand64(shape, seed, offset=0.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) + offset


def frame_mask(F, T, W, ref):
    f = np.arange(F)
    adj = np.abs(f[:, None] - f[None, :]) <= W
    if ref >= 0:
        adj[:, ref] = True
    return np.kron(adj, np.ones((T, T), dtype=bool))


def sdpa64(q, k, v, scale, mask=None):
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    am = None if mask is None else torch.from_numpy(mask)
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=am, scale=scale)
    return out.numpy()


def test_dense_equals_sdpa():
    """W >= F-1 reduces to ordinary dense softmax attention."""
    B, H, F, T, D = 1, 2, 5, 24, 32
    N = F * T
    q, k, v = (rand64((B, H, N, D), s) for s in (1, 2, 3))
    scale = D ** -0.5
    o, lse, _ = oracle.attention_rows(q, k, v, T, F - 1, 0, scale)
    want = sdpa64(q, k, v, scale).reshape(-1, D)
    np.testing.assert_allclose(o, want, atol=1e-12, rtol=0)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    np.testing.assert_allclose(lse, logsumexp(s, axis=-1).reshape(-1), atol=1e-12, rtol=0)


def test_block_diagonal_equals_per_frame_sdpa():
    """No reference frame and W = 0: each frame attends only to itself."""
    B, H, F, T, D = 1, 3, 4, 16, 16
    N = F * T
    q, k, v = (rand64((B, H, N, D), s) for s in (4, 5, 6))
    scale = 0.3
    o, _, _ = oracle.attention_rows(q, k, v, T, 0, -1, scale)
    o = o.reshape(B, H, N, D)
    for f in range(F):
        sl = slice(f * T, (f + 1) * T)
        want = sdpa64(q[:, :, sl], k[:, :, sl], v[:, :, sl], scale)
        np.testing.assert_allclose(o[:, :, sl], want, atol=1e-12, rtol=0)


@pytest.mark.parametrize("F,T,W,ref", [(4, 48, 1, 0), (7, 16, 2, 3), (6, 32, 1, -1), (9, 16, 1, 0)])
def test_sparse_equals_masked_sdpa(F, T, W, ref):
    B, H, D = 1, 2, 32
    N = F * T
    q, k, v = (rand64((B, H, N, D), s, off) for s, off in ((7, 0), (8, 0.5), (9, 0)))
    scale = D ** -0.5
    m = frame_mask(F, T, W, ref)
    o, lse, mx = oracle.attention_rows(q, k, v, T, W, ref, scale)
    np.testing.assert_allclose(o, sdpa64(q, k, v, scale, m).reshape(-1, D), atol=1e-12, rtol=0)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    s = np.where(m, s, -np.inf)
    np.testing.assert_allclose(lse, logsumexp(s, axis=-1).reshape(-1), atol=1e-12, rtol=0)
    np.testing.assert_allclose(mx, s.max(axis=-1).reshape(-1), atol=1e-12, rtol=0)


def test_bf16_inputs_are_read_exactly():
    """bf16 bit patterns and their exact float64 values give identical results."""
    w = configs.TINY
    q, k, v = synth.make_qkv(w)
    o1, l1, _ = oracle.attention_rows(q, k, v, w.T, w.W, w.ref, w.scale)
    o2, l2, _ = oracle.attention_rows(*(t.to(torch.float64) for t in (q, k, v)),
                                      w.T, w.W, w.ref, w.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_centring_invariance():
    """Subtracting the key mean shifts every logit of a row by the same amount,
    so the outputs are unchanged (exact arithmetic; fp64 to 1e-12)."""
    B, H, F, T, D = 1, 2, 5, 16, 32
    N = F * T
    q = rand64((B, H, N, D), 10)
    k = rand64((B, H, N, D), 11, offset=2.0)
    v = rand64((B, H, N, D), 12)
    c = k.mean(axis=2, keepdims=True)
    o1, _, _ = oracle.attention_rows(q, k, v, T, 1, 0, 0.2)
    o2, _, _ = oracle.attention_rows(q, k - c, v, T, 1, 0, 0.2)
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)


def test_permutation_within_frame():
    """Permuting keys (with their values) inside one frame leaves O unchanged."""
    B, H, F, T, D = 1, 2, 4, 32, 16
    N = F * T
    q, k, v = (rand64((B, H, N, D), s) for s in (13, 14, 15))
    perm = np.arange(N)
    rng = np.random.default_rng(0)
    perm[T:2 * T] = T + rng.permutation(T)
    o1, _, _ = oracle.attention_rows(q, k, v, T, 1, 0, 0.25)
    o2, _, _ = oracle.attention_rows(q, k[:, :, perm], v[:, :, perm], T, 1, 0, 0.25)
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("w", [configs.TINY, configs.SMALL.with_(F=5, T=48)])
def test_bound_at_least_true_max(w):
    """m_i >= max_{j in J(i)} s_ij for every row, under the windowed mask, for
    eligible and outlier heads alike ("Unchaining the Softmax": the bound's
    guarantee extends to windowed sparse masks)."""
    q, k, v = synth.make_qkv(w)
    st = oracle.key_stats(q, k, w.scale, 64.0)
    m = oracle.row_bounds(q, st["c"], st["R"], w.scale)
    _, _, mx = oracle.attention_rows(q, k, v, w.T, w.W, w.ref, w.scale)
    assert (m >= mx - 1e-12).all()
    # and the gap never exceeds the per-head G = 2 * scale * Qmax * R
    gap = (m - mx).reshape(w.B * w.H, -1)
    assert (gap <= st["G"].reshape(-1, 1) + 1e-12).all()


def test_bound_is_tight_for_aligned_key():
    """Closed form: if the key farthest from the mean points along q, the bound
    equals that key's logit exactly."""
    D = 8
    q = np.zeros((1, 1, 2, D)); q[0, 0, :, 0] = 2.0
    k = np.zeros((1, 1, 2, D)); k[0, 0, 0, 0] = 3.0; k[0, 0, 1, 0] = -3.0
    v = rand64((1, 1, 2, D), 1)
    st = oracle.key_stats(q, k, 0.5, 64.0)
    assert st["R"][0, 0] == pytest.approx(3.0) and np.allclose(st["c"], 0)
    m = oracle.row_bounds(q, st["c"], st["R"], 0.5)
    _, _, mx = oracle.attention_rows(q, k, v, 2, 0, -1, 0.5)   # one frame of 2 tokens
    np.testing.assert_allclose(m, [3.0, 3.0], atol=1e-15)
    np.testing.assert_allclose(mx, [3.0, 3.0], atol=1e-15)


def test_bound_closed_form_with_offset_mean():
    """Closed form with a non-zero key mean c: keys c +- a e0 and c +- a e1 have
    mean c and R = a. A query along e0 meets the Cauchy-Schwarz equality case, so
    its bound scale*(q.c + |q| a) equals its true max; a query along e2 sees the
    same logit scale*q.c on every key, so its bound exceeds its max by exactly
    scale*|q|*a. Both the q.c term and the |q| R term are needed to match."""
    D, a, scale = 8, 2.0, 0.5
    c = np.zeros(D); c[:3] = [1.5, -0.75, 0.5]
    k = np.tile(c, (1, 1, 4, 1))
    k[0, 0, 0, 0] += a; k[0, 0, 1, 0] -= a; k[0, 0, 2, 1] += a; k[0, 0, 3, 1] -= a
    q = np.zeros((1, 1, 4, D)); q[0, 0, 0, 0] = 2.0; q[0, 0, 1, 2] = 3.0
    q[0, 0, 2, 0] = -1.0; q[0, 0, 3, 1] = 0.5
    v = rand64((1, 1, 4, D), 2)
    st = oracle.key_stats(q, k, scale, 64.0)
    np.testing.assert_allclose(st["c"].reshape(-1), c, atol=0, rtol=0)
    assert st["R"][0, 0] == a
    m = oracle.row_bounds(q, st["c"], st["R"], scale)
    _, _, mx = oracle.attention_rows(q, k, v, 4, 0, -1, scale)   # one frame of 4 tokens
    qc = q[0, 0] @ c
    qn = np.linalg.norm(q[0, 0], axis=-1)
    np.testing.assert_allclose(m, scale * (qc + qn * a), atol=1e-15, rtol=0)
    # rows 0, 2, 3 point along a key axis (equality case); row 1 is orthogonal to both
    np.testing.assert_allclose(mx[[0, 2, 3]], m[[0, 2, 3]], atol=1e-15, rtol=0)
    assert mx[1] == pytest.approx(scale * qc[1], abs=1e-15)
    assert m[1] - mx[1] == pytest.approx(scale * 3.0 * a, abs=1e-15)


def test_static_max_equals_max_subtracted():
    """Softmax with the precomputed bound as the shift equals the ordinary
    max-subtracted softmax (the static-max reformulation is exact)."""
    w = configs.TINY
    q, k, v = synth.make_qkv(w)
    st = oracle.key_stats(q, k, w.scale, 64.0)
    m = oracle.row_bounds(q, st["c"], st["R"], w.scale).reshape(w.B, w.H, w.N)
    o, lse, _ = oracle.attention_rows(q, k, v, w.T, w.W, w.ref, w.scale)
    q64, k64, v64 = (synth.bf16_to_f64(t) for t in (q, k, v))
    s = w.scale * np.einsum("bhid,bhjd->bhij", q64, k64)
    mask = frame_mask(w.F, w.T, w.W, w.ref)
    p = np.where(mask, np.exp(s - m[..., None]), 0.0)
    l = p.sum(-1)
    o_static = np.einsum("bhij,bhjd->bhid", p, v64) / l[..., None]
    np.testing.assert_allclose(o_static.reshape(-1, w.D), o, atol=1e-12, rtol=0)
    np.testing.assert_allclose((m + np.log(l)).reshape(-1), lse, atol=1e-12, rtol=0)


def test_online_softmax_equals_definition():
    """Flash-style online softmax over key blocks (running max, rescale on every
    raise -- "Unchaining the Softmax") reproduces the plain definition."""
    w = configs.TINY
    q, k, v = synth.make_qkv(w)
    o, lse, _ = oracle.attention_rows(q, k, v, w.T, w.W, w.ref, w.scale)
    q64, k64, v64 = (synth.bf16_to_f64(t) for t in (q, k, v))
    mask = frame_mask(w.F, w.T, w.W, w.ref)
    bk = 16
    B, H, N, D = q64.shape
    out = np.zeros_like(q64)
    lse2 = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                mrun, l, acc = -np.inf, 0.0, np.zeros(D)
                for j0 in range(0, N, bk):
                    js = [j for j in range(j0, j0 + bk) if mask[i, j]]
                    if not js:
                        continue
                    s = w.scale * k64[b, h, js] @ q64[b, h, i]
                    mnew = max(mrun, s.max())
                    a = np.exp(mrun - mnew)
                    p = np.exp(s - mnew)
                    l = l * a + p.sum()
                    acc = acc * a + p @ v64[b, h, js]
                    mrun = mnew
                out[b, h, i] = acc / l
                lse2[b, h, i] = mrun + np.log(l)
    np.testing.assert_allclose(out.reshape(-1, D), o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse2.reshape(-1), lse, atol=1e-12, rtol=0)


def test_key_stats_match_numpy():
    w = configs.SMALL.with_(F=3, T=80)
    q, k, _ = synth.make_qkv(w)
    st = oracle.key_stats(q, k, w.scale, 64.0)
    q64, k64 = synth.bf16_to_f64(q), synth.bf16_to_f64(k)
    c = k64.mean(axis=2)
    R = np.linalg.norm(k64 - c[:, :, None, :], axis=-1).max(-1)
    qmax = np.linalg.norm(q64, axis=-1).max(-1)
    np.testing.assert_allclose(st["c"], c, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(st["R"], R, rtol=1e-13)
    np.testing.assert_allclose(st["qmax"], qmax, rtol=1e-13)
    np.testing.assert_allclose(st["G"], 2 * w.scale * qmax * R, rtol=1e-13)
    # the outlier head (x20 key) is the only ineligible one
    assert list(st["elig"][0]) == [1] * 7 + [0]


def test_key_stats_closed_forms():
    """Constant keys: mean = the key, R = 0, G = 0, eligible. Keys +/- a e_1:
    mean 0, R = a. Queries of norm 3: Qmax = 3; G = 2 * scale * 3 * a."""
    D, N = 16, 10
    k = np.tile(np.linspace(-1, 1, D), (1, 1, N, 1))
    q = np.zeros((1, 1, N, D)); q[..., 3] = 3.0
    st = oracle.key_stats(q, k, 0.25, 64.0)
    np.testing.assert_allclose(st["c"][0, 0], np.linspace(-1, 1, D), atol=1e-15)
    assert st["R"][0, 0] < 1e-14 and st["elig"][0, 0] == 1
    k2 = np.zeros((1, 1, N, D)); k2[0, 0, ::2, 0] = 5.0; k2[0, 0, 1::2, 0] = -5.0
    st = oracle.key_stats(q, k2, 0.25, 7.0)
    assert st["R"][0, 0] == pytest.approx(5.0) and st["qmax"][0, 0] == pytest.approx(3.0)
    assert st["G"][0, 0] == pytest.approx(7.5)
    assert st["elig"][0, 0] == 0       # 7.5 > 7
    st = oracle.key_stats(q, k2, 0.25, 7.5)
    assert st["elig"][0, 0] == 1       # G <= tau is inclusive


def test_workload_eligibility():
    """The synthetic workloads put their x20 outlier heads, and only those,
    outside the G <= 64 rule (tiny and small configs, all heads)."""
    for w in (configs.TINY, configs.SMALL):
        q, k, _ = synth.make_qkv(w)
        st = oracle.key_stats(q, k, w.scale, 64.0)
        want = np.ones((w.B, w.H), dtype=np.uint8)
        for h in w.outlier_heads:
            want[:, h] = 0
        assert (st["elig"] == want).all()
        assert (np.abs(st["G"] - 64.0) > 0.25 * 64.0).all()   # far from the threshold

"""Pins for the per-query-frame bound ("Unchaining the Softmax": the bound stays
valid under windowed masks, where rows of different frames attend to different
subsets of the keys). Checked against numpy on an independent frame construction,
against the per-head statistics, and by the bound >= true max invariant."""
import numpy as np
import pytest

import oracle
from block_sparse_video_frame_gb300 import configs, synth


def live_frames(F, W, ref):
    f = np.arange(F)
    adj = np.abs(f[:, None] - f[None, :]) <= W
    if ref >= 0:
        adj[:, ref] = True
    return adj


@pytest.mark.parametrize("w", [configs.TINY, configs.SMALL.with_(F=7, T=48),
                               configs.SMALL.with_(F=6, T=32, W=0, ref=-1),
                               configs.TINY.with_(F=5, T=32, W=4)], ids=lambda w: f"{w.name}-{w.F}-{w.W}")
def test_frame_stats_match_numpy(w):
    q, k, _ = synth.make_qkv(w)
    fs = oracle.frame_stats(q, k, w.T, w.W, w.ref, w.scale, 64.0)
    q64, k64 = synth.bf16_to_f64(q), synth.bf16_to_f64(k)
    c = k64.mean(axis=2, keepdims=True)
    kn = np.linalg.norm(k64 - c, axis=-1).reshape(w.B, w.H, w.F, w.T)    # per key frame
    qn = np.linalg.norm(q64, axis=-1).reshape(w.B, w.H, w.F, w.T)
    Rg = kn.max(-1)                                                        # [B, H, F] per key frame
    adj = live_frames(w.F, w.W, w.ref)
    Rf = np.stack([Rg[..., adj[f]].max(-1) for f in range(w.F)], axis=-1)
    np.testing.assert_allclose(fs["R"], Rf, rtol=1e-13)
    np.testing.assert_allclose(fs["qmax"], qn.max(-1), rtol=1e-13)
    np.testing.assert_allclose(fs["G"], 2 * w.scale * qn.max(-1) * Rf, rtol=1e-13)
    # never looser than the per-head statistics, equal to them where a frame sees every key
    st = oracle.key_stats(q, k, w.scale, 64.0)
    assert (fs["R"] <= st["R"][..., None] + 1e-12).all()
    assert np.allclose(fs["R"].max(-1), st["R"]) or not adj.all(axis=1).any()
    assert ((fs["elig"] >= st["elig"][..., None])).all()


def test_frame_bound_at_least_true_max():
    w = configs.SMALL.with_(F=7, T=48)
    q, k, v = synth.make_qkv(w)
    st = oracle.key_stats(q, k, w.scale, 64.0)
    fs = oracle.frame_stats(q, k, w.T, w.W, w.ref, w.scale, 64.0)
    m = oracle.row_bounds_frames(q, st["c"], fs["R"], w.T, w.scale)
    _, _, mx = oracle.attention_rows(q, k, v, w.T, w.W, w.ref, w.scale)
    assert (m >= mx - 1e-12).all()
    gap = (m - mx).reshape(w.B, w.H, w.F, w.T)
    assert (gap <= fs["G"][..., None] + 1e-12).all()
    # and it is at least as tight as the per-head bound on every row
    m_head = oracle.row_bounds(q, st["c"], st["R"], w.scale)
    assert (m <= m_head + 1e-12).all()


def test_outlier_frame_only_taints_frames_that_see_it():
    """Closed form: one huge key in frame g* makes only the query frames whose
    live set contains g* ineligible."""
    w = configs.SMALL.with_(F=9, T=32, W=1, ref=0, outlier_heads=())
    q, k, _ = synth.make_qkv(w)
    k = k.clone()
    gstar = 6
    k[0, 2, gstar * w.T + 5, :] *= 40
    fs = oracle.frame_stats(q, k, w.T, w.W, w.ref, w.scale, 64.0)
    adj = live_frames(w.F, w.W, w.ref)
    assert list(fs["elig"][0, 2]) == [0 if adj[f, gstar] else 1 for f in range(w.F)]
    assert fs["elig"][0, [h for h in range(w.H) if h != 2]].all()

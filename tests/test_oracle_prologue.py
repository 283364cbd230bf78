"""Pins for the oracle's fused pre-attention chain ("Layout Is the ABI": the chain
of normalisation, projections, rotary embeddings and head packing that feeds
attention). Checked against numpy (RMSNorm, matmul), a complex-number
formulation of the rotation, and the rotary embedding's defining properties."""
import numpy as np
import pytest

import oracle

EPS, BASE = 1e-6, 10000.0


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def case(B=1, N=40, C=64, H=2, D=16, seed=0):
    x = rand((B, N, C), seed)
    w = rand((3 * H * D, C), seed + 1, C ** -0.5)
    g = 1.0 + 0.1 * rand((C,), seed + 2)
    return x, w, g, H, D


def numpy_reference(x, w, g, H, D):
    """RMSNorm and projection with numpy; rotation as complex multiplication
    (u + i w) * exp(i a) on the pairs (i, i + D/2)."""
    B, N, C = x.shape
    y = x / np.sqrt((x ** 2).mean(-1, keepdims=True) + EPS) * g
    z = y @ w.T                                      # [B, N, 3HD]
    z = z.reshape(B, N, 3, H, D)
    n = np.arange(N)[None, :, None, None]
    t = BASE ** (-2.0 * np.arange(D // 2) / D)
    rot = np.exp(1j * n * t)                         # [1, N, 1, D/2]
    out = []
    for part in range(3):
        zp = z[:, :, part]                           # [B, N, H, D]
        if part < 2:
            cz = (zp[..., : D // 2] + 1j * zp[..., D // 2:]) * rot
            zp = np.concatenate([cz.real, cz.imag], axis=-1)
        out.append(zp.reshape(B * N, H, D))
    return out


def test_matches_numpy_and_complex_rotation():
    x, w, g, H, D = case(B=2)
    got = oracle.qkv_prologue(x, w, g, H, D, EPS, BASE)
    want = numpy_reference(x, w, g, H, D)
    for a, b in zip(got, want):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_rotation_is_identity_at_position_zero_and_keeps_norms():
    x, w, g, H, D = case()
    q, k, v = oracle.qkv_prologue(x, w, g, H, D, EPS, BASE)
    plain = (x / np.sqrt((x ** 2).mean(-1, keepdims=True) + EPS) * g) @ w.T
    plain = plain.reshape(x.shape[1], 3, H, D)
    np.testing.assert_allclose(q[0], plain[0, 0], atol=1e-12)
    np.testing.assert_allclose(k[0], plain[0, 1], atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), np.linalg.norm(plain[:, 0], axis=-1), rtol=1e-12)
    np.testing.assert_allclose(v, plain[:, 2], atol=1e-12)       # v is never rotated


def test_scores_depend_only_on_relative_position():
    """q_m . k_n after the rotary embedding depends only on m - n: give every
    position the same hidden state and compare shifted pairs."""
    C, H, D, N = 64, 2, 16, 50
    row = rand((C,), 7)
    x = np.tile(row, (1, N, 1))
    w = rand((3 * H * D, C), 8, C ** -0.5)
    g = np.ones(C)
    q, k, _ = oracle.qkv_prologue(x, w, g, H, D, EPS, BASE)
    for m, n, s in ((3, 1, 20), (10, 25, 13), (0, 40, 9)):
        a = (q[m] * k[n]).sum(-1)
        b = (q[m + s] * k[n + s]).sum(-1)
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_rmsnorm_closed_form():
    """A constant hidden row a * 1 normalises to sign(a) * gamma."""
    C, H, D = 32, 1, 8
    x = np.full((1, 3, C), -2.5)
    w = np.zeros((3 * H * D, C))
    for o in range(3 * H * D):
        w[o, o % C] = 1.0                           # z_o = y_(o mod C)
    g = np.linspace(0.5, 1.5, C)
    q, k, v = oracle.qkv_prologue(x, w, g, H, D, 0.0, BASE)
    np.testing.assert_allclose(v[0, 0], -g[2 * H * D % C + np.arange(D)], atol=1e-12)
    np.testing.assert_allclose(q[0, 0], -g[np.arange(D)], atol=1e-12)      # position 0: no rotation


@pytest.mark.parametrize("dtype", ["bf16"])
def test_bf16_inputs_read_exactly(dtype):
    import torch
    x, w, g, H, D = case()
    xb = torch.from_numpy(x).to(torch.bfloat16)
    wb = torch.from_numpy(w).to(torch.bfloat16)
    a = oracle.qkv_prologue(xb, wb, g, H, D, EPS, BASE)
    b = oracle.qkv_prologue(xb.double(), wb.double(), g, H, D, EPS, BASE)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)

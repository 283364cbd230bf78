"""Shared helpers for the GPU parity tests: row sampling and the tolerance
checks. The expected values always come from the fp64 oracle."""
import numpy as np
import torch

import oracle

# Tolerances for attention outputs against fp64 with bf16 inputs and fp32
# accumulation: max-abs 1e-2, mean-abs 1e-3; LSE 1e-3 absolute.
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_ABS = 1e-3


def stratified_rows(w, per_frame_random=13, seed=1234):
    """Flattened row indices ((b*H + h)*N + i): per (b, h, frame) the frame's
    first and last row, the first row of its last T % 128 rows and the row
    before it (a tail that a gathered tile may hold, and the last whole tile),
    and `per_frame_random` seeded uniform rows; per segment (rows sharing one
    key-run list: a frame, or the whole sequence when dense) the first row of
    its last 128-row tile, which is shifted to end at the segment's end."""
    rng = np.random.default_rng(seed)
    rows = []
    seg = w.N if w.dense else w.T
    for bh in range(w.B * w.H):
        picks = set()
        for f in range(w.F):
            lo, hi = f * w.T, (f + 1) * w.T
            picks.update((lo, hi - 1))
            if w.T % 128 and w.T > 128:
                picks.update((hi - w.T % 128, hi - w.T % 128 - 1))
            picks.update(int(x) for x in rng.integers(lo, hi, per_frame_random))
        for s0 in range(0, w.N, seg):
            picks.add(max(s0, s0 + seg - 128))
        rows.extend(bh * w.N + i for i in sorted(picks))
    return np.array(rows, dtype=np.int64)


def oracle_rows(w, q, k, v, rows=None):
    return oracle.attention_rows(q, k, v, w.T, w.W, w.ref, w.scale, rows)


def gather_rows(t, rows, N):
    """t: [B, H, N, D] or [B, H, N] CUDA tensor -> numpy float64 of the given flat rows."""
    if t.dim() == 4:
        flat = t.reshape(-1, t.shape[-1])
    else:
        flat = t.reshape(-1)
    idx = torch.from_numpy(rows).to(t.device)
    return flat.index_select(0, idx).double().cpu().numpy()


def check_close(o_gpu, o_ref, lse_gpu=None, lse_ref=None, what=""):
    err = np.abs(o_gpu - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: max-abs {err.max():.3e} > {O_MAX_ABS}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e} > {O_MEAN_ABS}"
    if lse_gpu is not None:
        e2 = np.abs(lse_gpu - lse_ref)
        assert e2.max() <= LSE_ABS, f"{what}: lse max-abs {e2.max():.3e} > {LSE_ABS}"
    return float(err.max()), float(err.mean())

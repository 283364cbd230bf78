"""Pins for the oracle's mask and block schedule ("Deleting the Mask", Fig. 3 of
"HeyGen x Google Cloud: Bringing Avatar IV to TPUs").

The schedule is pinned against (1) hand-derived closed-form counts stored in
tests/golden/schedule_counts.json, (2) an independent construction of the
token mask as a Kronecker product of a frame adjacency matrix with a T x T
block of ones, and (3) the pages' claim that block sizes dividing the frame
span leave no partially live block while 128-multiple tiles do not.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "schedule_counts.json")))
CASES = [(k, v) for k, v in GOLD.items() if not k.startswith("_")]


def frame_adjacency(F, W, ref):
    """F x F boolean: query frame f sees key frame g. Built from the distance
    matrix |f - g| (numpy broadcasting), independent of the C oracle."""
    f = np.arange(F)
    adj = np.abs(f[:, None] - f[None, :]) <= W
    if ref >= 0:
        adj[:, ref] = True
    return adj


def closed_form_frame_pairs(F, W, ref):
    total = 0
    for f in range(F):
        lo, hi = max(0, f - W), min(F - 1, f + W)
        total += hi - lo + 1
        if ref >= 0 and not (lo <= ref <= hi):
            total += 1
    return total


@pytest.mark.parametrize("name,c", CASES)
def test_closed_form_counts(name, c):
    assert closed_form_frame_pairs(c["F"], c["W"], c["ref"]) == c["frame_pairs"]
    assert frame_adjacency(c["F"], c["W"], c["ref"]).sum() == c["frame_pairs"]
    assert c["frame_pairs"] * c["T"] ** 2 == c["live_pairs_per_head"]


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_schedule_live_pairs_match_golden(name):
    c = GOLD[name]
    bs = 16
    s = oracle.schedule(c["F"], c["T"], c["W"], c["ref"], bs)
    assert s.live_pairs == c["live_pairs_per_head"]
    # every live block is full: nnz * bs^2 == live pairs
    assert len(s.col_idx) * bs * bs == c["live_pairs_per_head"]


def test_mask_brute_force_tiny():
    """Every token pair of the tiny case against the Kronecker-product mask."""
    F, T, W, ref = 4, 48, 1, 0
    N = F * T
    want = np.kron(frame_adjacency(F, W, ref), np.ones((T, T), dtype=bool))
    got = np.array([[oracle.mask(T, W, ref, i, j) for j in range(N)] for i in range(N)])
    assert (got == want).all()


@pytest.mark.parametrize("F,T,W,ref", [(4, 48, 1, 0), (9, 400, 1, 0), (6, 32, 0, -1),
                                       (7, 16, 2, 3), (5, 64, 4, 0), (8, 48, 1, 7)])
def test_schedule_csr_and_runs(F, T, W, ref):
    """CSR and per-frame runs equal what the frame adjacency implies."""
    adj = frame_adjacency(F, W, ref)
    for bs in [b for b in range(16, T + 1, 16) if T % b == 0]:
        s = oracle.schedule(F, T, W, ref, bs)
        per = T // bs
        blk = np.kron(adj, np.ones((per, per), dtype=bool))
        nb = F * per
        assert len(s.row_ptr) == nb + 1
        for qb in range(nb):
            cols = s.col_idx[s.row_ptr[qb]:s.row_ptr[qb + 1]]
            assert list(cols) == list(np.nonzero(blk[qb])[0])
        assert s.live_pairs == adj.sum() * T * T
        for f in range(F):
            live = np.nonzero(adj[f])[0]
            runs = []
            for g in live:  # maximal runs of consecutive frames, in tokens
                if runs and runs[-1][1] == g * T:
                    runs[-1][1] = (g + 1) * T
                else:
                    runs.append([g * T, (g + 1) * T])
            assert len(runs) <= 2
            want = runs[0] + (runs[1] if len(runs) > 1 else [0, 0])
            assert list(s.runs[f]) == want


def frame_level_census(F, T, W, ref, tile):
    """(full, partial, dead) tile x tile blocks from the frame adjacency alone: a
    block's token pairs are all live when every (query frame, key frame) pair it
    covers is adjacent, none when no pair is. Independent of the oracle's
    token-by-token count."""
    adj = frame_adjacency(F, W, ref)
    N = F * T
    edges = [(i0, min(i0 + tile, N)) for i0 in range(0, N, tile)]
    span = [(a // T, (b - 1) // T) for a, b in edges]
    counts = [0, 0, 0]
    for fa, fb in span:
        for ga, gb in span:
            sub = adj[fa:fb + 1, ga:gb + 1]
            counts[0 if sub.all() else (1 if sub.any() else 2)] += 1
    return tuple(counts)


def test_block_census_hand_counts():
    """Hand-derived censuses ("Deleting the Mask": tiles that straddle frame
    boundaries come out partial).
    (a) Two frames of 48 tokens, block-diagonal mask (W = 0, no reference), 32-token
        tiles: tiles 0 and 2 lie inside one frame each, tile 1 straddles both; the
        diagonal tiles (0,0) and (2,2) are full, (0,2) and (2,0) dead, the five
        pairs touching tile 1 partial.
    (b) Three frames of 48, W = 0, reference frame 0, 32-token tiles (the last one
        16 tokens): per query tile the counts are (1,1,3), (1,2,2), (3,0,2),
        (3,1,1), (3,1,1) as (full, partial, dead)."""
    assert oracle.block_census(2, 48, 0, -1, 32) == (2, 5, 2)
    assert oracle.block_census(3, 48, 0, 0, 32) == (11, 5, 9)


@pytest.mark.parametrize("F,T,W,ref,tile", [
    (9, 400, 1, 0, 128), (9, 400, 1, 0, 80), (4, 48, 1, 0, 128), (13, 120, 2, 0, 128),
    (13, 120, 2, 0, 1024), (7, 144, 1, 3, 256), (6, 160, 0, -1, 128), (21, 104, 20, 0, 128),
    (5, 37 * 16, 1, 4, 48),
])
def test_block_census_matches_frame_level_construction(F, T, W, ref, tile):
    got = oracle.block_census(F, T, W, ref, tile)
    assert got == frame_level_census(F, T, W, ref, tile)
    assert sum(got) == (-(-F * T // tile)) ** 2


def test_misaligned_blocks_are_partial():
    """Blocks of 128 tokens over frames whose token count 128 does not divide mix
    live and dead token pairs ("Deleting the Mask"): 128-token blocks over
    400-token frames leave partial blocks (the exact count from the frame-level
    construction), a divisor of the span leaves none."""
    F, T, W, ref = 9, 400, 1, 0
    full, partial, dead = oracle.block_census(F, T, W, ref, 128)
    assert (full, partial, dead) == frame_level_census(F, T, W, ref, 128)
    assert partial > 0
    with pytest.raises(ValueError):
        oracle.schedule(F, T, W, ref, 128)
    full, partial, dead = oracle.block_census(F, T, W, ref, 80)
    assert partial == 0 and full * 80 * 80 == frame_adjacency(F, W, ref).sum() * T * T


def test_dense_ragged_blocks_all_live():
    """W >= F-1 is dense: every block (including a ragged last one) is live."""
    F, T = 5, 24  # N = 120, bs = 16 leaves a ragged 8-token block
    s = oracle.schedule(F, T, F - 1, 0, 16)
    nb = (F * T + 15) // 16
    assert len(s.col_idx) == nb * nb
    assert s.live_pairs == (F * T) ** 2
    assert (s.runs == np.array([0, F * T, 0, 0])).all()

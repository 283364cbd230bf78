"""GPU parity of the block schedule ("Deleting the Mask", Fig. 3): CSR, per-frame
key runs, nnz and live pairs are bit-exact against the oracle, which tests every
token pair of every block through the token-level mask."""
import numpy as np
import pytest
import torch

import oracle
import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs

pytestmark = pytest.mark.gpu

CASES = [
    (4, 48, 1, 0, 16), (4, 48, 1, 0, 48),          # tiny
    (9, 400, 1, 0, 16), (9, 400, 1, 0, 80),        # small
    (13, 3600, 2, 0, 240), (13, 3600, 2, 0, 144),  # 720p-like
    (9, 8160, 1, 0, 240),                          # 1080p-like
    (21, 1560, 20, 0, 16), (21, 1560, 20, 0, 128), # dense base DiT (ragged last block)
    (7, 16, 2, 3, 16), (6, 32, 0, -1, 32), (1, 64, 0, 0, 16), (8, 48, 1, 7, 16),
    (5, 24, 4, 0, 16), (12, 32, 3, -1, 16),
    (1, 1, 0, 0, 16), (5, 8, 4, 0, 16), (3, 5, 2, -1, 16),   # one token; tiny dense sequences
    (9, 1040, 1, 0, 80), (6, 1072, 2, 5, 16), (5, 1088, 1, -1, 64),  # gathered tails of 16, 48, 64 rows
]


@pytest.mark.parametrize("F,T,W,ref,bs", CASES)
def test_schedule_bit_exact(F, T, W, ref, bs):
    plan = vd.attn_plan(F, T, W, ref, bs)
    want = oracle.schedule(F, T, W, ref, bs)
    torch.cuda.synchronize()
    assert plan.info.live_pairs == want.live_pairs
    assert plan.info.nnz == len(want.col_idx)
    assert np.array_equal(plan.row_ptr().cpu().numpy(), want.row_ptr)
    assert np.array_equal(plan.col_idx().cpu().numpy(), want.col_idx)
    assert np.array_equal(plan.frame_runs().cpu().numpy(), want.runs)
    plan.rebuild()
    assert np.array_equal(plan.col_idx().cpu().numpy(), want.col_idx)


@pytest.mark.parametrize("F,T,W,ref,bs", CASES)
def test_work_units_cover_every_query_row_once(F, T, W, ref, bs):
    """Host-logic check of the attention work list: every query row is owned by
    exactly one 128-row tile: a tile of a unit (a pair of its segment's tiles), a
    gathered tile, or a tail tile. Segments group frames with equal key runs. A
    gathered tile holds the ragged last rows of 2 to 8 segments (multiples of 16,
    at most 64 each, 128 in all) and visits the union of their key runs, at least
    a quarter smaller than the runs the tails would each visit alone; only
    segments of at least 1024 rows give up their tails. A plan without gathered
    tiles and with at least 32 tile pairs per head hands the tiles of the last 8
    pairs of its last unit class's last segment to the second launch as one-tile
    records. The units of a segment are its first tile pairs, ordered by
    non-increasing key count, one count per cost class."""
    plan = vd.attn_plan(F, T, W, ref, bs)
    runs = plan.frame_runs().cpu().numpy()
    segs = plan.segments().cpu().numpy()
    units = plan.units().cpu().numpy()
    cls = plan.class_offsets().cpu().numpy()
    gat = plan.gathers().cpu().numpy()
    N = F * T
    covered = np.zeros(N, dtype=np.int64)

    def own(s, t):   # rows tile t of segment s owns (the last tile is shifted to end at the end)
        row0, rows = int(s[0]), int(s[1])
        return row0 + 128 * t, row0 + min(128 * (t + 1), rows)

    gathered_seg, tail = set(), []
    multi = [g for g in gat if g[0] >= 2]
    for g in gat:
        npc, rows, lo0, hi0, lo1, hi1, one, keys = (int(x) for x in g[:8])
        assert 1 <= npc <= 8 and one == 1 and 0 < rows <= 128
        assert keys == (hi0 - lo0) + (hi1 - lo1) and lo0 < hi0 and (hi1 == lo1 == 0 or hi0 < lo1 < hi1)
        if npc == 1:   # a tail tile: one tile of a segment, the rows it owns
            sg, r0, nr = (int(x) for x in g[8:11])
            s = segs[sg]
            t = (r0 - int(s[0])) // 128
            assert len(multi) == 0 and (r0 - int(s[0])) % 128 == 0 and (r0, r0 + nr) == own(s, t)
            assert [lo0, hi0, lo1, hi1] == [int(x) for x in s[2:6]] and keys == int(s[7])
            covered[r0:r0 + nr] += 1
            tail.append((sg, t))
            continue
        live = np.zeros(N, dtype=bool)
        live[lo0:hi0] = True
        live[lo1:hi1] = True
        total, sum_keys = 0, 0
        for k in range(npc):
            sg, r0, nr = (int(x) for x in g[8 + 3 * k:11 + 3 * k])
            s = segs[sg]
            assert nr == s[1] % 128 and nr % 16 == 0 and nr <= 64 and r0 == s[0] + s[1] - nr
            assert s[1] >= 1024
            assert live[s[2]:s[3]].all() and live[s[4]:s[5]].all()
            covered[r0:r0 + nr] += 1
            total += nr
            sum_keys += int(s[7])
            gathered_seg.add(sg)
        assert total == rows and 4 * keys <= 3 * sum_keys
    for si, s in enumerate(segs):
        row0, rows, lo0, hi0, lo1, hi1, ntile, keys = (int(x) for x in s)
        f0 = row0 // T
        for f in range(f0, f0 + rows // T):
            assert list(runs[f]) == [lo0, hi0, lo1, hi1]
        assert keys == (hi0 - lo0) + (hi1 - lo1)
        assert ntile == (rows // 128 if si in gathered_seg else (rows + 127) // 128)
    seen = {}
    for code in units:
        idx, pair = int(code) >> 16, int(code) & 0xFFFF
        seen[(idx, pair)] = seen.get((idx, pair), 0) + 1
        s = segs[idx]
        for t in (2 * pair, 2 * pair + 1):
            if t < s[6]:
                lo, hi = own(s, t)
                covered[lo:hi] += 1
    assert all(c == 1 for c in seen.values())
    assert (covered == 1).all()
    # the units of a segment are its first tile pairs; the tail tiles are the rest of one segment
    for si, s in enumerate(segs):
        ps = sorted(p for (i, p) in seen if i == si)
        assert ps == list(range(len(ps)))
    if tail:
        sg = tail[0][0]
        ts = sorted(t for _, t in tail)
        npairs = (int(segs[sg][6]) + 1) // 2
        kept = len([1 for (i, _) in seen if i == sg])
        assert all(x == sg for x, _ in tail) and ts == list(range(2 * kept, int(segs[sg][6])))
        assert npairs - kept == min(8, npairs - 1) and len(units) + npairs - kept >= 32
        assert units[-1] >> 16 == sg   # the last unit class's last segment
    keys = np.array([segs[int(c) >> 16][7] for c in units])
    assert (np.diff(keys) <= 0).all()
    assert cls[0] == 0 and cls[-1] == len(units)
    for a, b in zip(cls[:-1], cls[1:]):
        assert len(set(keys[a:b])) == 1


def host_second_launch_records(F, T, W, ref):
    """The records of the second attention launch, restated on the host from the
    rule in vdit.h: segments are runs of frames with equal key runs; tails
    (rows % 128, a multiple of 16, at most 64, of segments of at least 1024 rows
    that see keys) are packed greedily in segment order into groups of at most 8
    pieces and 128 rows whose key runs unite into at most two runs; a group of
    two or more whose union has at most 3/4 of the pieces' keys is a gathered
    tile. Without gathered tiles and with at least 32 tile pairs per head, the
    tiles of the last 8 pairs (keeping one) of the last segment in unit order
    (stable, by non-increasing key count) become one-piece tail tiles. Returns
    the records as lists of 32 ints and the tile count of each segment."""
    def runs_of(f):
        lo, hi = max(0, f - W), min(F - 1, f + W)
        r = [lo * T, (hi + 1) * T, 0, 0]
        if ref >= 0 and not lo <= ref <= hi:
            if ref == lo - 1:
                r[0] = ref * T
            elif ref == hi + 1:
                r[1] = (ref + 1) * T
            elif ref < lo:
                r = [ref * T, (ref + 1) * T, lo * T, (hi + 1) * T]
            else:
                r = [lo * T, (hi + 1) * T, ref * T, (ref + 1) * T]
        return r

    segs = []                      # [row0, rows, runs]
    for f in range(F):
        r = runs_of(f)
        if segs and segs[-1][2] == r:
            segs[-1][1] += T
        else:
            segs.append([f * T, T, r])
    ntile = [(rows + 127) // 128 for _, rows, _ in segs]
    keys = [(r[1] - r[0]) + (r[3] - r[2]) for _, _, r in segs]

    def union(a, b):
        iv = sorted(x for x in [(a[0], a[1]), (a[2], a[3]), (b[0], b[1]), (b[2], b[3])] if x[1] > x[0])
        m = []
        for lo, hi in iv:
            if m and lo <= m[-1][1]:
                m[-1] = (m[-1][0], max(m[-1][1], hi))
            else:
                m.append((lo, hi))
        if len(m) > 2:
            return None
        m += [(0, 0)] * (2 - len(m))
        return [m[0][0], m[0][1], m[1][0], m[1][1]]

    recs, group, gr, grows, gkeys = [], [], [0, 0, 0, 0], 0, 0

    def close():
        nonlocal group, gr, grows, gkeys
        uk = (gr[1] - gr[0]) + (gr[3] - gr[2])
        if len(group) >= 2 and 4 * uk <= 3 * gkeys:
            rec = [len(group), grows] + gr + [1, uk]
            for sg, r0, nr in group:
                rec += [sg, r0, nr]
                ntile[sg] = segs[sg][1] // 128
            recs.append(rec + [0] * (32 - len(rec)))
        group, gr, grows, gkeys = [], [0, 0, 0, 0], 0, 0

    for sg, (row0, rows, r) in enumerate(segs):
        tail = rows % 128
        if keys[sg] == 0 or rows < 1024 or tail == 0 or tail % 16 or tail > 64:
            continue
        u = union(gr, r)
        if group and not (u is not None and len(group) < 8 and grows + tail <= 128):
            close()
            u = union(gr, r)
        group.append((sg, row0 + rows - tail, tail))
        gr, grows, gkeys = u, grows + tail, gkeys + keys[sg]
    close()
    if not recs:
        order = sorted(range(len(segs)), key=lambda i: -keys[i])   # stable
        used = [i for i in order if keys[i] > 0]
        pairs = [(ntile[i] + 1) // 2 for i in used]
        if used and sum(pairs) >= 32:
            sg = used[-1]
            npairs = (ntile[sg] + 1) // 2
            mv = min(8, npairs - 1)
            row0, rows, r = segs[sg]
            for t in range(2 * (npairs - mv), ntile[sg]):
                own = min(128, rows - 128 * t)
                rec = [1, own] + r + [1, keys[sg], sg, row0 + 128 * t, own]
                recs.append(rec + [0] * (32 - len(rec)))
    return recs, ntile


@pytest.mark.parametrize("F,T,W,ref,bs", CASES + [(4096, 1040, 2, 0, 1040), (5, 1660, 4, 0, 16),
                                                 (4, 8160, 1, 0, 240)])
def test_second_launch_records_follow_the_rule(F, T, W, ref, bs):
    """The device plan's gathered and tail tiles, and its segments' tile counts,
    equal a host restatement of the packing rule, field by field."""
    plan = vd.attn_plan(F, T, W, ref, bs)
    want, ntile = host_second_launch_records(F, T, W, ref)
    got = plan.gathers().cpu().numpy()
    # fields past the pieces are not written by the plan: compare the used ones
    assert len(got) == len(want)
    for g, w in zip(got, want):
        n = 8 + 3 * w[0]
        assert [int(x) for x in g[:n]] == w[:n]
    assert [int(x) for x in plan.segments().cpu().numpy()[:, 6]] == ntile


def test_gathered_tiles_of_the_720p_geometry():
    """13 frames of 3600 tokens (28 whole tiles and a 16-row tail each), window
    +-2 and reference frame 0: the tails of frames 0-7 share one tile over frames
    0-9, those of frames 8-12 one over frames 6-12 plus frame 0; every segment
    keeps 28 tiles."""
    T = 3600
    plan = vd.attn_plan(13, T, 2, 0, 240)
    segs = plan.segments().cpu().numpy()
    gat = plan.gathers().cpu().numpy()
    assert len(segs) == 13 and (segs[:, 6] == 28).all()
    assert gat.shape == (2, 32)
    assert list(gat[0, :8]) == [8, 128, 0, 10 * T, 0, 0, 1, 10 * T]
    assert list(gat[1, :8]) == [5, 80, 0, T, 6 * T, 13 * T, 1, 8 * T]
    for gi, frames in ((0, range(0, 8)), (1, range(8, 13))):
        pieces = gat[gi, 8:8 + 3 * len(frames)].reshape(-1, 3)
        assert [tuple(x) for x in pieces] == [(f, f * T + 3584, 16) for f in frames]
    assert plan.info.n_units == 13 * 14 and plan.info.n_gathers == 2


def test_segment_at_the_tile_pair_field_limit():
    """Maximum size of the work-unit encoding (segment << 16 | tile pair): a
    dense sequence of exactly 2^24 rows holds 65 536 tile pairs in the 16-bit
    pair field (the last 8 of them handed to the second launch as tail tiles);
    one more 128-row tile is refused as unsupported instead of wrapping into the
    segment field."""
    T = 1 << 24
    plan = vd.attn_plan(1, T, 0, 0, 4096)
    units = plan.units().cpu().numpy().astype(np.int64)
    # the last 8 pairs' 16 tiles run as tail tiles in the second launch
    assert plan.info.n_segments == 1 and len(units) == 65536 - 8 and plan.info.n_gathers == 16
    assert (units >> 16 == 0).all()
    assert np.array_equal(units & 0xFFFF, np.arange(65536 - 8))
    gat = plan.gathers().cpu().numpy()
    assert [int(g[9]) for g in gat] == [128 * t for t in range(2 * 65528, 2 * 65536)]
    assert plan.info.live_pairs == T * T
    plan.close()
    with pytest.raises(vd.VditError) as ei:
        vd.attn_plan(1, T + 128, 0, 0, 4096)
    assert ei.value.status == vd.VDIT_ERR_UNSUPPORTED
    assert "tile pairs" in str(ei.value)


def test_plan_at_the_frame_limit():
    """The largest plan in frames (4096, the meta kernel's per-frame arrays), with
    16-token frames, window +-2 and reference frame 0. Expected values come from
    the window rule itself: per frame the clipped window [f-2, f+2] plus frame 0
    when it lies outside; one segment and one 16-row tile per frame (segments this
    short keep their tails: no gathered tile); units of one cost class per key
    count."""
    F, T, W, ref, bs = 4096, 16, 2, 0, 16
    plan = vd.attn_plan(F, T, W, ref, bs)
    frames = []
    for f in range(F):
        lo, hi = max(0, f - W), min(F - 1, f + W)
        runs = [[lo * T, (hi + 1) * T]]
        if not lo <= ref <= hi:
            runs = ([[ref * T, (ref + 1) * T], [lo * T, (hi + 1) * T]] if lo > ref + 1
                    else [[ref * T, (hi + 1) * T]])
        frames.append(runs[0] + (runs[1] if len(runs) > 1 else [0, 0]))
    want_runs = np.array(frames, dtype=np.int32)
    assert np.array_equal(plan.frame_runs().cpu().numpy(), want_runs)
    keys = [(r[1] - r[0]) + (r[3] - r[2]) for r in frames]
    assert plan.info.live_pairs == sum(keys) * T
    assert plan.info.nnz == sum(keys) // bs
    segs = plan.segments().cpu().numpy()
    units = plan.units().cpu().numpy().astype(np.int64)
    assert plan.info.n_segments == F and len(units) == F and plan.info.n_gathers == 0
    assert sorted(int(s[0]) for s in segs) == [f * T for f in range(F)]
    # longest first: the unit key counts never increase, and each class has one count
    ukeys = np.array([segs[u >> 16][7] for u in units])
    assert (np.diff(ukeys) <= 0).all()
    assert sorted(ukeys.tolist(), reverse=True) == sorted(keys, reverse=True)
    cls = plan.class_offsets().cpu().numpy()
    assert len(cls) - 1 == len(set(keys))


def test_gathered_tiles_at_the_frame_limit():
    """4096 frames of 1040 tokens (8 whole tiles and a 16-row tail each), window
    +-2 and reference frame 0: frames 8g..8g+7 share gathered tile g, over the
    union of their windows and frame 0, and every segment keeps its 8 tiles."""
    F, T, W, ref, bs = 4096, 1040, 2, 0, 1040
    plan = vd.attn_plan(F, T, W, ref, bs)
    segs = plan.segments().cpu().numpy()
    assert plan.info.n_segments == F and (segs[:, 6] == 8).all()
    assert plan.info.n_units == 4 * F
    gat = plan.gathers().cpu().numpy()
    assert gat.shape == (F // 8, 32)
    for g in range(F // 8):
        lo, hi = max(0, 8 * g - W), min(F - 1, 8 * g + 7 + W)
        union = [0, (hi + 1) * T, 0, 0] if lo <= ref + 1 else [0, T, lo * T, (hi + 1) * T]
        ukeys = (union[1] - union[0]) + (union[3] - union[2])
        assert list(gat[g, :8]) == [8, 128] + union + [1, ukeys]
        want = [(f, f * T + 1024, 16) for f in range(8 * g, 8 * g + 8)]
        assert [tuple(x) for x in gat[g, 8:].reshape(-1, 3)] == want


CENSUS = [
    (9, 400, 1, 0, 80, 128), (9, 400, 1, 0, 80, 80),        # small: 128-tiles vs a divisor
    (4, 48, 1, 0, 16, 128), (4, 48, 1, 0, 16, 16),           # tiny
    (13, 3600, 2, 0, 240, 128), (13, 3600, 2, 0, 240, 1024),  # 720p-like
    (9, 8160, 1, 0, 240, 128), (9, 8160, 1, 0, 240, 1024),    # 1080p-like
    (21, 1560, 20, 0, 16, 128),                               # dense: every block live
    (3, 48, 0, 0, 16, 32), (2, 48, 0, -1, 16, 32), (7, 144, 1, 3, 48, 256),
]


@pytest.mark.parametrize("F,T,W,ref,bs,tile", CENSUS)
def test_block_census_bit_exact(F, T, W, ref, bs, tile):
    """Partial blocks under a frame-blind tiling ("Deleting the Mask": about one
    live block in five partial under 128-multiple tiles), counted on the device,
    equal the oracle's token-by-token count."""
    plan = vd.attn_plan(F, T, W, ref, bs)
    got = plan.block_census(tile)
    assert got == oracle.block_census(F, T, W, ref, tile)
    if T % tile == 0:
        assert got[1] == 0

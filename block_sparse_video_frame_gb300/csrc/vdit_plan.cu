// Block schedule of the frame-window + reference-frame mask.
//
// "HeyGen x Google Cloud: Bringing Avatar IV to TPUs", "Deleting the Mask"
// (Fig. 3): a query in frame f sees the keys of frames g with |f - g| <= W
// (clipped to the sequence) plus the reference frame. With a block size that
// is a multiple of 16 and divides the frame's token span, each block is either
// entirely live or entirely dead, and the reference frame contributes
// ordinary live blocks to the same pass.
//
// Two kernels build the plan on the device:
//   plan_meta_kernel  per-frame key runs (at most two maximal runs of live key
//                     tokens: the window and, when outside it, the reference
//                     frame), segments of consecutive frames sharing one run
//                     list, the attention kernel's work units ordered longest
//                     first, and the header counts (nnz, live pairs).
//   plan_csr_kernel   the CSR of live (query block, key block) pairs.
#include <cuda_runtime.h>

#include <cstdlib>
#include <new>

#include "vdit_internal.h"

namespace vdit {
namespace {

struct PlanArgs {
    int F, T, W, ref, bs, dense, part;
    long long N;
    int nqb;
    int units_cap;
};

// Window [wlo, whi] of frame f and whether the reference frame adds a run.
__device__ __forceinline__ void frame_window(const PlanArgs &a, int f, int &wlo, int &whi) {
    wlo = f - a.W < 0 ? 0 : f - a.W;
    whi = f + a.W > a.F - 1 ? a.F - 1 : f + a.W;
}

// Live key frames of frame f, as at most two maximal token runs [lo, hi).
// Part 1 keeps the window alone, part 2 the reference frame alone (for frames
// whose window does not contain it; other frames see no key).
__device__ void frame_runs_of(const PlanArgs &a, int f, int r[4], int &live_frames) {
    int wlo, whi;
    frame_window(a, f, wlo, whi);
    long long T = a.T;
    const int g = a.ref;
    const bool ref_outside = g >= 0 && (g < wlo || g > whi);
    if (a.part == VDIT_PART_REFERENCE) {
        live_frames = ref_outside ? 1 : 0;
        r[0] = ref_outside ? (int)(g * T) : 0;
        r[1] = ref_outside ? (int)((g + 1) * T) : 0;
        r[2] = 0; r[3] = 0;
        return;
    }
    live_frames = whi - wlo + 1;
    int lo0 = (int)(wlo * T), hi0 = (int)((whi + 1) * T), lo1 = 0, hi1 = 0;
    if (ref_outside && a.part == VDIT_PART_ALL) {
        live_frames += 1;
        if (g == wlo - 1) {
            lo0 = (int)(g * T);                       // adjacent below: merge
        } else if (g == whi + 1) {
            hi0 = (int)((g + 1) * T);                 // adjacent above: merge
        } else if (g < wlo) {
            lo1 = lo0; hi1 = hi0;                     // reference run first
            lo0 = (int)(g * T); hi0 = (int)((g + 1) * T);
        } else {
            lo1 = (int)(g * T); hi1 = (int)((g + 1) * T);
        }
    }
    r[0] = lo0; r[1] = hi0; r[2] = lo1; r[3] = hi1;
}

// Union of a gathered tile's key runs r (empty runs have hi <= lo) with a
// segment's runs s, written to u as at most two ascending runs; false when the
// union needs more than two. Every index is fixed at compile time (a sorting
// network, then an unrolled merge), so the arrays stay in registers.
__device__ __forceinline__ bool union_runs(const int r[4], const int s[4], int u[4]) {
    constexpr int kNone = 0x7fffffff;   // an empty run sorts last
    int lo[4] = {r[0], r[2], s[0], s[2]}, hi[4] = {r[1], r[3], s[1], s[3]};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (hi[i] <= lo[i]) lo[i] = hi[i] = kNone;
    auto cswap = [&](int i, int j) {
        if (lo[j] < lo[i]) {
            const int tl = lo[i], th = hi[i];
            lo[i] = lo[j]; hi[i] = hi[j];
            lo[j] = tl; hi[j] = th;
        }
    };
    cswap(0, 1); cswap(2, 3); cswap(0, 2); cswap(1, 3); cswap(1, 2);
    int m = 0, ml[2] = {0, 0}, mh[2] = {0, 0};
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (lo[i] == kNone) continue;
        if (m > 0 && lo[i] <= (m == 1 ? mh[0] : mh[1])) {
            if (m == 1) mh[0] = max(mh[0], hi[i]);
            else mh[1] = max(mh[1], hi[i]);
        } else if (m < 2) {
            if (m == 0) { ml[0] = lo[i]; mh[0] = hi[i]; }
            else { ml[1] = lo[i]; mh[1] = hi[i]; }
            ++m;
        } else {
            ok = false;
        }
    }
    u[0] = ml[0]; u[1] = mh[0]; u[2] = ml[1]; u[3] = mh[1];
    return ok;
}

// One block. The frames' runs are computed in parallel; one thread then builds
// the segments, packs their ragged last rows into gathered tiles, sorts the
// segments and lays out the cost classes, with every intermediate in shared
// memory (the runs of a frame are recomputed, not read back); the unit list is
// written by all threads.
__global__ void plan_meta_kernel(PlanArgs a, PlanHeader *__restrict__ hdr, int32_t *__restrict__ frame_runs,
                                 int32_t *__restrict__ segments, int32_t *__restrict__ units,
                                 int32_t *__restrict__ class_off, int32_t *__restrict__ gathers) {
    // s_cnt: live frames per frame, then per segment its key count, then its first unit.
    // s_order: segments longest first, each entry (tile pairs << 12) | segment.
    __shared__ int s_cnt[kMaxFrames];
    __shared__ int s_order[kMaxFrames];
    __shared__ int s_nused;   // entries of s_order that get units
    __shared__ int s_pseg[kGatherMaxPieces], s_prows[kGatherMaxPieces];
    static_assert(kMaxFrames <= (1 << 12), "segment index field of s_order");
    for (int f = threadIdx.x; f < a.F; f += blockDim.x) {
        int r[4], live;
        frame_runs_of(a, f, r, live);
        frame_runs[4 * f + 0] = r[0];
        frame_runs[4 * f + 1] = r[1];
        frame_runs[4 * f + 2] = r[2];
        frame_runs[4 * f + 3] = r[3];
        s_cnt[f] = live;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        PlanHeader h{};
        // counts ------------------------------------------------------------
        long long fp = 0;
        for (int f = 0; f < a.F; ++f) fp += s_cnt[f];
        h.live_pairs = fp * (long long)a.T * a.T;
        if (a.dense) {
            h.nnz = (long long)a.nqb * a.nqb;
        } else {
            long long per = a.T / a.bs;
            h.nnz = fp * per * per;
        }
        // segments: consecutive frames with identical run lists, and gathered
        // tiles ---------------------------------------------------------------
        // A segment whose row count is not a multiple of 128 ends in a tile that
        // holds only its last rows % 128 rows. Consecutive such tails (multiples
        // of 16 rows, at most kGatherMaxRows each) of segments with at least 8
        // whole tiles are packed into one 128-row tile that visits the union of
        // their key runs, when that union is at most two runs and at least a
        // quarter smaller than the key runs the tails would each visit in a tile
        // of their own; the segments then keep only their whole tiles. (Shorter
        // segments give a launch too little work to hide the gathered tiles,
        // whose key runs are longer than any of theirs.) The gathered tiles are
        // not work units: a second launch of the attention kernel runs them.
        // Everything the packing reads is in registers or shared memory (s_pseg,
        // s_prows: the open tile's pieces).
        int nseg = 0, cur[4] = {0, 0, 0, 0}, row0 = 0, rows = 0;
        int ng = 0, npc = 0, grows = 0, gr[4] = {0, 0, 0, 0};
        long long sum_keys = 0;
        auto close = [&]() {
            const long long ukeys = (long long)(gr[1] - gr[0]) + (gr[3] - gr[2]);
            if (npc >= 2 && 4 * ukeys <= 3 * sum_keys) {
                int32_t *rec = gathers + kGatherInts * ng;
                rec[0] = npc; rec[1] = grows;
                rec[2] = gr[0]; rec[3] = gr[1]; rec[4] = gr[2]; rec[5] = gr[3];
                rec[6] = 1; rec[7] = (int)ukeys;
                for (int k = 0; k < npc; ++k) {
                    const int sg = s_pseg[k], nt = s_prows[k] / kTileRows;
                    segments[kSegInts * sg + 6] = nt;
                    s_order[sg] = (min((nt + kTilesPerUnit - 1) / kTilesPerUnit, kMaxPairsPerSegment) << 12) | sg;
                }
                ++ng;
            }
            npc = 0; grows = 0; sum_keys = 0;
            gr[0] = gr[1] = gr[2] = gr[3] = 0;
        };
        auto add_tail = [&](int sg, int keys) {
            const int tail = rows % kTileRows;
            if (keys == 0 || rows < kGatherMinSegRows || tail == 0 || tail % 16 != 0 || tail > kGatherMaxRows)
                return;
            int u[4];
            const bool joins = union_runs(gr, cur, u) && npc < kGatherMaxPieces && grows + tail <= kTileRows;
            if (npc > 0 && !joins) {
                close();
                union_runs(gr, cur, u);
            }
            int32_t *pc = gathers + kGatherInts * ng + kGatherPiece + 3 * npc;
            pc[0] = sg; pc[1] = row0 + rows - tail; pc[2] = tail;
            s_pseg[npc] = sg;
            s_prows[npc] = rows;
            gr[0] = u[0]; gr[1] = u[1]; gr[2] = u[2]; gr[3] = u[3];
            grows += tail;
            sum_keys += keys;
            ++npc;
        };
        auto flush = [&]() {
            int32_t *g = segments + kSegInts * nseg;
            const int ntile = (rows + kTileRows - 1) / kTileRows;
            const int keys = (cur[1] - cur[0]) + (cur[3] - cur[2]);
            const int npairs = (ntile + kTilesPerUnit - 1) / kTilesPerUnit;
            g[0] = row0; g[1] = rows;
            g[2] = cur[0]; g[3] = cur[1]; g[4] = cur[2]; g[5] = cur[3];
            g[6] = ntile; g[7] = keys;
            // a unit code keeps the tile pair in its low 16 bits
            if (npairs > kMaxPairsPerSegment) h.error = 4;
            s_cnt[nseg] = keys;        // frame counts are no longer needed
            s_order[nseg] = (min(npairs, kMaxPairsPerSegment) << 12) | nseg;
            add_tail(nseg, keys);
            ++nseg;
        };
        for (int f = 0; f < a.F; ++f) {
            int r[4], live;
            frame_runs_of(a, f, r, live);
            if (f > 0 && r[0] == cur[0] && r[1] == cur[1] && r[2] == cur[2] && r[3] == cur[3]) {
                rows += a.T;
                continue;
            }
            if (f > 0) flush();
            cur[0] = r[0]; cur[1] = r[1]; cur[2] = r[2]; cur[3] = r[3];
            row0 = (int)((long long)f * a.T);
            rows = a.T;
        }
        flush();
        close();
        if (h.error != 0) nseg = ng = 0;
        // longest first (stable insertion sort on key count) ------------------
        for (int i = 1; i < nseg; ++i) {
            const int v = s_order[i], key = s_cnt[v & 0xFFF];
            int j = i - 1;
            while (j >= 0 && s_cnt[s_order[j] & 0xFFF] < key) {
                s_order[j + 1] = s_order[j];
                --j;
            }
            s_order[j + 1] = v;
        }
        // tail tiles ---------------------------------------------------------
        // A plan without gathered tiles hands the last kTailPairs tile pairs of
        // its last segment in this order (the shortest units, which a launch runs
        // last) to the chained second launch, as one-tile records of one piece
        // each (the rows the tile owns). That launch's CTAs take the SMs the tile
        // pairs free at their end one tile at a time. Only plans with at least
        // kTailMinPairs tile pairs per head do this: a launch with less work has
        // no long tail to fill.
        if (ng == 0 && h.error == 0) {
            int total = 0, last = -1;
            for (int i = 0; i < nseg; ++i) {
                const int v = s_order[i];
                if (s_cnt[v & 0xFFF] == 0) break;
                total += v >> 12;
                if ((v >> 12) > 0) last = i;
            }
            if (last >= 0 && total >= kTailMinPairs) {
                const int v = s_order[last], sg = v & 0xFFF, np = v >> 12;
                const int mv = min(kTailPairs, np - 1);   // the segment keeps at least one pair
                const int32_t *g = segments + kSegInts * sg;
                const int srow0 = g[0], srows = g[1], ntile = g[6];
                for (int t = 2 * (np - mv); t < ntile; ++t) {
                    int32_t *rec = gathers + kGatherInts * ng;
                    const int own = min(kTileRows, srows - kTileRows * t);
                    rec[0] = 1; rec[1] = own;
                    rec[2] = g[2]; rec[3] = g[3]; rec[4] = g[4]; rec[5] = g[5];
                    rec[6] = 1; rec[7] = g[7];
                    rec[kGatherPiece] = sg; rec[kGatherPiece + 1] = srow0 + kTileRows * t;
                    rec[kGatherPiece + 2] = own;
                    ++ng;
                }
                s_order[last] = ((np - mv) << 12) | sg;
            }
        }
        // cost classes and the first unit of each segment ---------------------
        int nu = 0, ncls = 0, prev_key = -1, i = 0;
        for (; i < nseg; ++i) {
            const int v = s_order[i], sg = v & 0xFFF, np = v >> 12, key = s_cnt[sg];
            if (key == 0) break;   // frames that see no key (reference part only): no work, sorted last
            if (np == 0) continue; // every row of the segment went to gathered tiles
            if (key != prev_key) {
                if (ncls >= kMaxClasses) { h.error = 2; break; }
                class_off[ncls++] = nu;
                prev_key = key;
            }
            if (nu + np > a.units_cap) { h.error = 3; break; }
            s_cnt[sg] = nu;
            nu += np;
        }
        class_off[ncls] = nu;
        h.n_segments = nseg;
        h.n_units = nu;
        h.n_classes = ncls;
        h.n_gathers = ng;
        *hdr = h;
        s_nused = i;
    }
    __syncthreads();
    // units: (segment << 16) | tile pair, in the order of s_order ------------
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
    for (int i = warp; i < s_nused; i += nwarps) {
        const int v = s_order[i], sg = v & 0xFFF, np = v >> 12, first = s_cnt[sg];
        for (int p = lane; p < np; p += 32) units[first + p] = (sg << 16) | p;
    }
}

// One warp per query block: the lanes sum the blocks of the earlier frames (the
// row's offset) and write the row's key blocks, 32 at a time.
__global__ void plan_csr_kernel(PlanArgs a, const int32_t *frame_runs, int32_t *row_ptr,
                                int32_t *col_idx) {
    const int qb = (int)((blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32);
    const int lane = threadIdx.x % 32;
    if (qb >= a.nqb) return;
    long long start, len;
    if (a.dense) {
        start = (long long)qb * a.nqb;
        len = a.nqb;
        for (int kb = lane; kb < a.nqb; kb += 32) col_idx[start + kb] = kb;
    } else {
        const int per = a.T / a.bs;
        const int f = qb / per;
        long long before = 0;
        for (int g = lane; g < f; g += 32) {
            const int32_t *r = frame_runs + 4 * g;
            before += (long long)((r[1] - r[0]) + (r[3] - r[2])) / a.bs;
        }
        for (int o = 16; o > 0; o /= 2) before += __shfl_xor_sync(0xffffffffu, before, o);
        const int32_t *r = frame_runs + 4 * f;
        const int n0 = (r[1] - r[0]) / a.bs, k0 = r[0] / a.bs, k1 = r[2] / a.bs;
        len = n0 + (r[3] - r[2]) / a.bs;
        start = before * per + (long long)(qb - f * per) * len;
        for (int i = lane; i < len; i += 32) col_idx[start + i] = i < n0 ? k0 + i : k1 + (i - n0);
    }
    if (lane == 0) {
        row_ptr[qb] = (int32_t)start;
        if (qb == a.nqb - 1) row_ptr[a.nqb] = (int32_t)(start + len);
    }
}

// Census of the tile x tile grid over the N x N token pairs (the last tile of
// each axis ragged when tile does not divide N): a tile is full when every
// token pair in it is live, dead when none is, partial otherwise. The mask
// depends only on the frames of the two tokens, so a tile is classified from
// the frame pairs it covers. One thread per tile, block-wide sums, three
// atomics per block.
__global__ void census_kernel(int F, int T, int W, int ref, long long N, int tile, long long nb,
                              unsigned long long *counts) {
    __shared__ unsigned long long s_cnt[3];
    if (threadIdx.x < 3) s_cnt[threadIdx.x] = 0;
    __syncthreads();
    unsigned long long c[3] = {0, 0, 0};
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < nb * nb;
         t += (long long)gridDim.x * blockDim.x) {
        const long long qb = t / nb, kb = t % nb;
        const long long i0 = qb * tile, i1 = min(i0 + tile, N);
        const long long j0 = kb * tile, j1 = min(j0 + tile, N);
        const int fa = (int)(i0 / T), fb = (int)((i1 - 1) / T);
        const int ga = (int)(j0 / T), gb = (int)((j1 - 1) / T);
        bool all = true, any = false;
        for (int f = fa; f <= fb; ++f)
            for (int g = ga; g <= gb; ++g) {
                const int d = f > g ? f - g : g - f;
                const bool live = d <= W || g == ref;
                all = all && live;
                any = any || live;
            }
        c[all ? 0 : (any ? 1 : 2)] += 1;
    }
    for (int i = 0; i < 3; ++i) {
        unsigned long long v = c[i];
        for (int o = 16; o > 0; o /= 2) v += __shfl_down_sync(0xffffffffu, v, o);
        if ((threadIdx.x & 31) == 0 && v) atomicAdd(&s_cnt[i], v);
    }
    __syncthreads();
    if (threadIdx.x < 3 && s_cnt[threadIdx.x]) atomicAdd(&counts[threadIdx.x], s_cnt[threadIdx.x]);
}

PlanArgs args_of(const vdit_plan *p) {
    PlanArgs a;
    a.F = p->F; a.T = p->T; a.W = p->W; a.ref = p->ref; a.bs = p->bs; a.dense = p->dense; a.part = p->part;
    a.N = p->N; a.nqb = p->n_qblocks; a.units_cap = p->units_cap;
    return a;
}

void free_plan_buffers(vdit_plan *p) {
    cudaFree(p->d_header);
    cudaFree(p->d_row_ptr);
    cudaFree(p->d_col_idx);
    cudaFree(p->d_frame_runs);
    cudaFree(p->d_segments);
    cudaFree(p->d_units);
    cudaFree(p->d_class_off);
    cudaFree(p->d_gathers);
    cudaFree(p->d_status);
}

}  // namespace

cudaError_t launch_plan_kernels(const vdit_plan *p, cudaStream_t stream, bool csr) {
    PlanArgs a = args_of(p);
    plan_meta_kernel<<<1, 256, 0, stream>>>(a, p->d_header, p->d_frame_runs, p->d_segments,
                                             p->d_units, p->d_class_off, p->d_gathers);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !csr) return e;
    plan_csr_kernel<<<(a.nqb + 7) / 8, 256, 0, stream>>>(a, p->d_frame_runs, p->d_row_ptr, p->d_col_idx);
    return cudaGetLastError();
}

}  // namespace vdit

using namespace vdit;

namespace {

vdit_status plan_create(int32_t F, int32_t T, int32_t W, int32_t ref, int32_t bs, int32_t part,
                        void *stream, vdit_plan **out) {
    clear_error();
    if (!out) { set_error("vdit_attn_plan: out is NULL"); return VDIT_ERR_INVALID; }
    *out = nullptr;
    if (F < 1 || F > kMaxFrames) {
        set_error("vdit_attn_plan: num_frames=%d outside [1, %d]", F, kMaxFrames);
        return VDIT_ERR_INVALID;
    }
    if (T < 1) { set_error("vdit_attn_plan: tokens_per_frame=%d < 1", T); return VDIT_ERR_INVALID; }
    if ((long long)F * T >= (1ll << 31)) {
        set_error("vdit_attn_plan: N = F*T = %lld does not fit int32", (long long)F * T);
        return VDIT_ERR_INVALID;
    }
    if (W < 0) { set_error("vdit_attn_plan: window_radius=%d < 0", W); return VDIT_ERR_INVALID; }
    if (ref < -1 || ref >= F) {
        set_error("vdit_attn_plan: ref_frame=%d outside [-1, %d]", ref, F - 1);
        return VDIT_ERR_INVALID;
    }
    if (bs < 16 || bs % 16 != 0) {
        set_error("vdit_attn_plan: block_size=%d is not a positive multiple of 16", bs);
        return VDIT_ERR_INVALID;
    }
    const int dense = W >= F - 1 ? 1 : 0;
    if (part != VDIT_PART_ALL && part != VDIT_PART_WINDOW && part != VDIT_PART_REFERENCE) {
        set_error("vdit_attn_plan_part: part=%d invalid", part);
        return VDIT_ERR_INVALID;
    }
    if (part != VDIT_PART_ALL && (dense || ref < 0)) {
        set_error("vdit_attn_plan_part: the mask has no separate reference part (%s)",
                  dense ? "the window covers every frame" : "no reference frame");
        return VDIT_ERR_INVALID;
    }
    if (!dense && T % bs != 0) {
        set_error("vdit_attn_plan: block_size=%d does not divide tokens_per_frame=%d "
                  "(blocks would straddle frame boundaries)", bs, T);
        return VDIT_ERR_INVALID;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    vdit_plan *p = new (std::nothrow) vdit_plan();
    if (!p) { set_error("vdit_attn_plan: host allocation failed"); return VDIT_ERR_NOMEM; }
    p->F = F; p->T = T; p->W = W; p->ref = ref; p->bs = bs; p->dense = dense; p->part = part;
    p->N = (long long)F * T;
    p->n_qblocks = (int)((p->N + bs - 1) / bs);
    p->units_cap = (int)(p->N / (kTileRows * kTilesPerUnit)) + 2 * F + 2;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "cudaGetDevice"); }
    e = device_alloc(reinterpret_cast<void **>(&p->d_header), sizeof(PlanHeader));
    if (e == cudaSuccess) e = device_alloc(reinterpret_cast<void **>(&p->d_frame_runs), sizeof(int32_t) * 4 * F);
    if (e == cudaSuccess) e = device_alloc(reinterpret_cast<void **>(&p->d_segments), sizeof(int32_t) * kSegInts * F);
    if (e == cudaSuccess) e = device_alloc(reinterpret_cast<void **>(&p->d_units), sizeof(int32_t) * p->units_cap);
    if (e == cudaSuccess) e = device_alloc(reinterpret_cast<void **>(&p->d_class_off), sizeof(int32_t) * (kMaxClasses + 1));
    // a gathered tile holds at least two segments' rows; or the plan has tail tiles
    if (e == cudaSuccess)
        e = device_alloc(reinterpret_cast<void **>(&p->d_gathers),
                         sizeof(int32_t) * kGatherInts * (F / 2 + 1 + kTilesPerUnit * kTailPairs));
    if (e == cudaSuccess) e = device_alloc(reinterpret_cast<void **>(&p->d_status), sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemsetAsync(p->d_status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) {
        free_plan_buffers(p);
        delete p;
        set_error("vdit_attn_plan: device allocation failed (%s)", cudaGetErrorString(e));
        return VDIT_ERR_NOMEM;
    }
    e = launch_plan_kernels(p, s, false);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&p->h, p->d_header, sizeof(PlanHeader),
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        free_plan_buffers(p);
        delete p;
        return cuda_fail(e, "vdit_attn_plan: schedule kernel");
    }
    if (p->h.error == 4) {
        set_error("vdit_attn_plan: a run of frames with equal key runs holds more than %d query rows "
                  "(%d tile pairs), beyond the work-unit encoding",
                  kMaxPairsPerSegment * kTileRows * kTilesPerUnit, kMaxPairsPerSegment);
        free_plan_buffers(p);
        delete p;
        return VDIT_ERR_UNSUPPORTED;
    }
    if (p->h.error != 0 || p->h.nnz >= (1ll << 31)) {
        set_error("vdit_attn_plan: schedule too large (error %d, nnz %lld)", p->h.error, p->h.nnz);
        free_plan_buffers(p);
        delete p;
        return VDIT_ERR_INVALID;
    }
    e = device_alloc(reinterpret_cast<void **>(&p->d_row_ptr), sizeof(int32_t) * (p->n_qblocks + 1));
    if (e == cudaSuccess) e = device_alloc(reinterpret_cast<void **>(&p->d_col_idx), sizeof(int32_t) * (p->h.nnz > 0 ? p->h.nnz : 1));
    if (e != cudaSuccess) {
        free_plan_buffers(p);
        delete p;
        set_error("vdit_attn_plan: device allocation failed (%s)", cudaGetErrorString(e));
        return VDIT_ERR_NOMEM;
    }
    e = launch_plan_kernels(p, s, true);
    if (e != cudaSuccess) {
        free_plan_buffers(p);
        delete p;
        return cuda_fail(e, "vdit_attn_plan: schedule kernels");
    }
    *out = p;
    return VDIT_OK;
}

}  // namespace

extern "C" vdit_status vdit_attn_plan(int32_t F, int32_t T, int32_t W, int32_t ref, int32_t bs,
                                      void *stream, vdit_plan **out) {
    return plan_create(F, T, W, ref, bs, VDIT_PART_ALL, stream, out);
}

extern "C" vdit_status vdit_attn_plan_part(int32_t F, int32_t T, int32_t W, int32_t ref, int32_t bs,
                                           int32_t part, void *stream, vdit_plan **out) {
    return plan_create(F, T, W, ref, bs, part, stream, out);
}

extern "C" vdit_status vdit_plan_rebuild(vdit_plan *p, void *stream) {
    clear_error();
    if (!p) { set_error("vdit_plan_rebuild: plan is NULL"); return VDIT_ERR_INVALID; }
    cudaError_t e = launch_plan_kernels(p, static_cast<cudaStream_t>(stream), true);
    if (e != cudaSuccess) return cuda_fail(e, "vdit_plan_rebuild");
    return VDIT_OK;
}

extern "C" vdit_status vdit_plan_get_info(const vdit_plan *p, vdit_plan_info *info) {
    clear_error();
    if (!p || !info) { set_error("vdit_plan_get_info: NULL argument"); return VDIT_ERR_INVALID; }
    info->num_frames = p->F;
    info->tokens_per_frame = p->T;
    info->window_radius = p->W;
    info->ref_frame = p->ref;
    info->block_size = p->bs;
    info->dense = p->dense;
    info->num_tokens = p->N;
    info->n_qblocks = p->n_qblocks;
    info->nnz = p->h.nnz;
    info->live_pairs = p->h.live_pairs;
    info->n_segments = p->h.n_segments;
    info->n_units = p->h.n_units;
    info->n_classes = p->h.n_classes;
    info->part = p->part;
    info->n_gathers = p->h.n_gathers;
    info->d_gathers = p->d_gathers;
    info->d_row_ptr = p->d_row_ptr;
    info->d_col_idx = p->d_col_idx;
    info->d_frame_runs = p->d_frame_runs;
    info->d_segments = p->d_segments;
    info->d_units = p->d_units;
    info->d_class_off = p->d_class_off;
    return VDIT_OK;
}

extern "C" vdit_status vdit_plan_status(vdit_plan *p, void *stream, int32_t *code) {
    clear_error();
    if (!p) { set_error("vdit_plan_status: plan is NULL"); return VDIT_ERR_INVALID; }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    VDIT_CUDA_TRY(cudaMemcpyAsync(&word, p->d_status, sizeof word, cudaMemcpyDeviceToHost, s));
    VDIT_CUDA_TRY(cudaStreamSynchronize(s));
    if (code) *code = word;
    if (word != 0) {
        VDIT_CUDA_TRY(cudaMemsetAsync(p->d_status, 0, sizeof(int32_t), s));
        VDIT_CUDA_TRY(cudaStreamSynchronize(s));
        set_error("a kernel's bounded wait expired (site code %d)", word);
        return VDIT_ERR_TIMEOUT;
    }
    return VDIT_OK;
}

extern "C" void vdit_plan_destroy(vdit_plan *p) {
    if (!p) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    free_plan_buffers(p);
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    delete p;
}

extern "C" vdit_status vdit_plan_block_census(const vdit_plan *p, int32_t tile, int64_t *counts,
                                              void *stream) {
    clear_error();
    if (!p || !counts) { set_error("vdit_plan_block_census: NULL argument"); return VDIT_ERR_INVALID; }
    if (tile < 16 || tile % 16 != 0) {
        set_error("vdit_plan_block_census: tile=%d is not a positive multiple of 16", tile);
        return VDIT_ERR_INVALID;
    }
    if ((reinterpret_cast<uintptr_t>(counts) & 7u) != 0) {
        set_error("vdit_plan_block_census: counts must be 8-byte aligned");
        return VDIT_ERR_INVALID;
    }
    const long long nb = (p->N + tile - 1) / tile;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    VDIT_CUDA_TRY(cudaMemsetAsync(counts, 0, 3 * sizeof(int64_t), s));
    const long long tiles = nb * nb;
    const int threads = 256;
    const long long blocks = (tiles + threads - 1) / threads;
    census_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), threads, 0, s>>>(
        p->F, p->T, p->W, p->ref, p->N, tile, nb, reinterpret_cast<unsigned long long *>(counts));
    VDIT_CUDA_TRY(cudaGetLastError());
    return VDIT_OK;
}

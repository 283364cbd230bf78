// Fused frame-window + reference-frame block-sparse attention for sm_103a.
//
// "HeyGen x Google Cloud: Bringing Avatar IV to TPUs":
//   "Deleting the Mask" (Fig. 3) -- the live key set of a query frame is at
//     most two runs of whole frames (the window and the reference frame), so
//     every key tile is fully live: no mask predicate, no padding, one pass.
//   "Unchaining the Softmax" (Fig. 4) -- on eligible heads each row's max is
//     fixed up front to m_i = scale * (q_i . c + |q_i| R) (Cauchy-Schwarz on
//     mean-centred keys), so p = 2^(s*log2e - m~) needs no running max and no
//     rescale of the accumulator; other heads run online softmax in the same
//     kernel (head-uniform branch).
//   "Proving the Pixels Didn't Change" -- P is rounded to bf16 and the final
//     P.V product runs on the matrix unit.
//
// GB300 design. Persistent grid (one CTA per SM, 320 threads):
//   warp 0          TMEM allocator and tcgen05.mma issuer (the warp walks the
//                   schedule, one elected lane issues)
//   warp 1          TMA producer: Q tiles, then a 2-stage ring of K tiles and a
//                   3-stage ring of V tiles (128 keys x D, bf16, 128-byte swizzle)
//   warps 2-5, 6-9  softmax warpgroups, one per 128-row query tile; thread t
//                   of a warpgroup owns TMEM lane t = query row t (warp w reads
//                   the lane quarter w % 4)
// A work unit is (b, h, segment, pair of query tiles); the CTAs walk them two
// heads at a time (see decode). Both tiles of a unit
// lie in one segment (frames with identical key runs), share every K/V tile
// and ping-pong on the tensor core:
//   S0 = Q0 K_0^T, S1 = Q1 K_0^T, then for each key tile j:
//   O0 += P0_j V_j, S0 = Q0 K_{j+1}^T, O1 += P1_j V_j, S1 = Q1 K_{j+1}^T
// so one warpgroup's exponentials overlap the other's MMAs. TMEM (512 cols):
// O0 | O1 | S0 | S1; P (bf16, two per 32-bit column) overwrites the first half
// of its S buffer and is the A operand (from TMEM) of the P.V MMA.
// A segment with an odd number of tiles ends in a lone tile. Its key tiles
// alternate between both slots (both read the same Q tile), so it overlaps like
// a pair; the epilogue adds O0 + O1 and the two row sums, exact because both
// halves share the static bound (online: both halves rescaled to the larger of
// their two running maxima first).
// A segment whose rows are not a multiple of 128 leaves a short last tile. The
// plan packs such tails of several segments into gathered tiles (each row masked
// to its own key runs), or, in a plan without those, hands the tiles of its last
// tile pairs over as one-tile records ("tail tiles"); a second instance of this
// kernel runs these records, launched as a programmatic dependent of the first
// so that its CTAs take the SMs the first one's CTAs leave at its end.
// Every wait is bounded in time; on expiry the CTA records a site code in the
// plan's status word, drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "vdit_internal.h"
#include "vdit_ptx.cuh"

namespace vdit {
namespace {

using namespace ptx;

constexpr int kBK = 128;              // keys per K/V tile
constexpr int kStagesK = 2;           // K ring depth (a K tile is free once its S MMAs finish)
constexpr int kStagesV = 3;           // V ring depth (V is held until P.V finishes)
constexpr int kThreads = 320;
constexpr int kWarpTma = 1;
constexpr int kWarpMma = 0;
constexpr int kWarpSoftmax0 = 2;      // softmax warpgroups: warps 2-5 and 6-9
constexpr int kHalfBytes = 128 * 128; // 128 rows x 64 bf16 (one swizzle-atom column)
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;
constexpr float kLazyRescale = 8.0f;  // online: rescale only when the max rises > 2^8
// Compile-time loop: f(std::integral_constant<int, i>) for i in [0, N).
template <int N, int I = 0, typename F>
__device__ __forceinline__ void static_for(F &&f) {
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for<N, I + 1>(f);
    }
}

// kernel instances: the frame-aligned tiles of the plan, the frame-blind tiling
// of the design before frame alignment, the plan's gathered tiles
enum : int { kModeAligned = 0, kModeTiled = 1, kModeGathered = 2 };

// status-word site codes (which wait expired)
enum : int {
    kSiteQfree = 1, kSiteKfree, kSiteVfree, kSiteQfullMma, kSiteKfull, kSiteVfull, kSitePfull,
    kSiteOfree, kSiteQfullSm, kSiteSfull, kSiteOfull, kSiteDrain, kSiteXfull, kSiteXfree
};

template <int D>
struct Layout {
    static constexpr int kTileBytes = kTileRows * D * 2;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTilesPerUnit * kTileBytes;
    static constexpr int kV = kK + kStagesK * kTileBytes;
    static constexpr int kBar = kV + kStagesV * kTileBytes;
    static constexpr int kX = kBar + 256;          // row sums and maxima handed between warpgroups
    static constexpr int kBytes = kX + kTileRows * 8;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
    static constexpr uint32_t kTmemO = 0;         // O0 at col 0, O1 at col D
    static constexpr uint32_t kTmemS = 2 * D;     // S0 at 2D, S1 at 2D + 128
};

// barrier slots (8 bytes each) after the tiles
enum : int {
    kBarQfull = 0, kBarQfree = 1, kBarKfull = 2, kBarKfree = kBarKfull + kStagesK,
    kBarVfull = kBarKfree + kStagesK, kBarVfree = kBarVfull + kStagesV,
    kBarSfull = kBarVfree + kStagesV, kBarPfull = kBarSfull + 2, kBarOfull = kBarPfull + 2,
    kBarOfree = kBarOfull + 2, kBarFinal = kBarOfree + 2,
    kBarXfull = kBarFinal + 1, kBarXfree = kBarXfull + 1, kNumBars = kBarXfree + 1
};
// the barriers, the TMEM address word and the abort flag share the 256 bytes at kBar
static_assert(8 * kNumBars + 8 <= 256, "barrier block overflows its 256 bytes");

struct Params {
    const int32_t *segments, *units, *class_off;
    int n_classes;
    int B, H, N;
    long long total_work;
    void *o;
    long long os0, os1, os2;
    int o_f32;
    float *lse;
    float scale_log2;  // scale * log2(e)
    const float *k_mean, *k_rmax;
    const uint8_t *elig;
    const float *seg_rmax;       // per (b, h, segment) bound and eligibility, or null
    const uint8_t *seg_elig;
    int nseg;
    int mode;
    int *status;
    unsigned long long timeout_ns;
    // frame-blind tiling (ablation of the design before frame alignment): the
    // mask's geometry, which part of it runs, and the 256-row query blocks per head
    int F, T, W, ref, part;
    int n_blocks;
    // gathered tiles: [n_gathers] records of the plan
    const int32_t *gathers;
    int n_gathers;
};

struct Work {
    int b, h, bh;
    int row0, rows;        // segment rows
    int lo0, hi0, lo1, hi1;
    int seg, pair, ntile;  // segment, this unit's tile pair, tiles in the segment
    int nact;              // active query tiles (1 or 2)
    int nt0, nkt;          // key tiles of run 0, total key tiles
    bool stat;             // static-max softmax (else online)
    bool alt;              // lone static tile: slots 0 and 1 take alternate key tiles
    int gat;               // gathered tile: its record
};

// Work order. CTA b takes work items b, b + grid, b + 2*grid, ... The items walk
// the heads in groups of kHeadGroup. Inside a group they walk the plan's cost
// classes longest first, and inside a class every head of the group with its
// units. So the CTAs running at one time share the K/V of at most a few heads,
// which stay in L2 (24 MB per head at 720p, D = 128). A head-major walk would
// still revisit each head's K/V once per cost class, after it has left L2.
constexpr int kHeadGroup = 2;

__device__ __forceinline__ void decode(const Params &p, long long w, Work &u) {
    const int BH = p.B * p.H;
    const long long per_head = p.class_off[p.n_classes];
    const long long g = w / (per_head * kHeadGroup);
    const int gh = min(kHeadGroup, BH - (int)g * kHeadGroup);   // heads in this group
    w -= g * per_head * kHeadGroup;
    long long base = 0;
    int c = 0, n_c = 0;
    for (c = 0; c < p.n_classes; ++c) {
        n_c = p.class_off[c + 1] - p.class_off[c];
        const long long span = (long long)n_c * gh;
        if (w < base + span) break;
        base += span;
    }
    const long long local = w - base;
    u.bh = (int)(g * kHeadGroup + local / n_c);
    const int ui = p.class_off[c] + (int)(local % n_c);
    u.b = u.bh / p.H;
    u.h = u.bh % p.H;
    const int code = p.units[ui];
    const int32_t *s = p.segments + kSegInts * (code >> 16);
    u.pair = code & 0xFFFF;
    u.seg = code >> 16;
    u.row0 = s[0]; u.rows = s[1];
    u.lo0 = s[2]; u.hi0 = s[3]; u.lo1 = s[4]; u.hi1 = s[5];
    u.ntile = s[6];
    u.nact = min(kTilesPerUnit, u.ntile - kTilesPerUnit * u.pair);
    u.nt0 = (u.hi0 - u.lo0 + kBK - 1) / kBK;
    u.nkt = u.nt0 + (u.hi1 - u.lo1 + kBK - 1) / kBK;
    u.stat = p.mode == VDIT_MODE_FORCE_STATIC ||
             (p.mode == VDIT_MODE_AUTO &&
              (p.seg_elig ? p.seg_elig[(size_t)u.bh * p.nseg + u.seg] : p.elig[u.bh]) != 0);
    // A lone tile has no partner to overlap its softmax with. Its key tiles
    // alternate between both slots (even ones in slot 0, odd ones in slot 1, both
    // reading the same Q tile). On the static path the bound is common to both
    // halves, so O = O0 + O1 and l = l0 + l1 exactly, with no rescale; online,
    // each half keeps its own running max and the epilogue rescales both halves
    // to the larger one.
    u.alt = u.nact == 1 && u.nkt >= 2;
}

// The design before frame alignment ("Deleting the Mask", Fig. 3): query blocks
// of 256 rows (two 128-row tiles) and 128-key tiles at fixed multiples of 128
// over the sequence padded to a multiple of 128, blind to frame boundaries. A
// block visits every 128-key tile that holds a live key of one of its rows: the
// window of its first to last frame and, when some row's window leaves it out,
// the reference frame (each rounded out to 128 keys); tiles where a row also
// sees dead keys are masked element by element in the softmax. Row i of the
// padded tail (i >= N) is computed as a row of the last frame and not stored.
// Blocks walk the heads in order, each head's blocks in sequence order.
__device__ __forceinline__ void decode_tiled(const Params &p, long long w, Work &u) {
    const long long per_head = p.n_blocks;
    u.bh = (int)(w / per_head);          // heads in order, blocks in sequence order inside a head
    const int blk = (int)(w % per_head);
    u.b = u.bh / p.H;
    u.h = u.bh % p.H;
    const int npad = (p.N + kBK - 1) / kBK * kBK;
    u.seg = 0;
    u.pair = 0;
    u.row0 = blk * kTilesPerUnit * kTileRows;
    u.rows = min(kTilesPerUnit * kTileRows, npad - u.row0);
    u.ntile = u.rows / kTileRows;
    u.nact = u.ntile;
    const int T = p.T;
    const int fa = u.row0 / T, fb = (min(u.row0 + u.rows, p.N) - 1) / T;
    const int wlo = max(0, fa - p.W), whi = min(p.F - 1, fb + p.W);
    // some row of the block has the reference frame outside its window
    const bool ref_needed = p.ref >= 0 && (p.ref < fb - p.W || p.ref > fa + p.W);
    int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    if (p.part != VDIT_PART_REFERENCE) { lo0 = wlo * T; hi0 = (whi + 1) * T; }
    if (p.part != VDIT_PART_WINDOW && ref_needed && (p.part == VDIT_PART_REFERENCE || p.ref < wlo || p.ref > whi)) {
        lo1 = p.ref * T;
        hi1 = (p.ref + 1) * T;
    }
    auto round_out = [&](int &lo, int &hi) {
        if (hi > lo) { lo = lo / kBK * kBK; hi = min((hi + kBK - 1) / kBK * kBK, npad); }
    };
    round_out(lo0, hi0);
    round_out(lo1, hi1);
    if (hi0 <= lo0) { lo0 = lo1; hi0 = hi1; lo1 = hi1 = 0; }          // the reference run alone
    if (hi1 > lo1) {
        if (lo1 < lo0) { int t0 = lo0, t1 = hi0; lo0 = lo1; hi0 = hi1; lo1 = t0; hi1 = t1; }
        if (lo1 <= hi0) { hi0 = max(hi0, hi1); lo1 = hi1 = 0; }        // overlapping after rounding
    }
    u.lo0 = lo0; u.hi0 = hi0; u.lo1 = lo1; u.hi1 = hi1;
    u.nt0 = (hi0 - lo0) / kBK;
    u.nkt = u.nt0 + (hi1 - lo1) / kBK;
    u.stat = p.mode == VDIT_MODE_FORCE_STATIC || (p.mode == VDIT_MODE_AUTO && p.elig[u.bh] != 0);
    u.alt = u.nact == 1 && u.nkt >= 2;
}

// Gathered tiles (the second launch): item w is record w % n_gathers of head
// B*H - 1 - w / n_gathers, last head first: the tile pairs end on the last heads,
// whose K/V are then still in L2. One query tile, whose rows come from up to 8
// segments, over the union of their key runs; with per-segment bounds it takes
// the static path only if every piece's segment may.
__device__ __forceinline__ void decode_gathered(const Params &p, long long w, Work &u) {
    u.bh = p.B * p.H - 1 - (int)(w / p.n_gathers);
    u.gat = (int)(w % p.n_gathers);
    u.b = u.bh / p.H;
    u.h = u.bh % p.H;
    const int32_t *g = p.gathers + kGatherInts * u.gat;
    u.seg = -1;
    u.pair = 0;
    u.row0 = 0; u.rows = g[1];
    u.lo0 = g[2]; u.hi0 = g[3]; u.lo1 = g[4]; u.hi1 = g[5];
    u.ntile = 1;
    u.nact = 1;
    u.nt0 = (u.hi0 - u.lo0 + kBK - 1) / kBK;
    u.nkt = u.nt0 + (u.hi1 - u.lo1 + kBK - 1) / kBK;
    // the eligibility arrays are read in AUTO mode only (they may be null otherwise)
    bool elig = p.mode == VDIT_MODE_AUTO;
    if (elig && !p.seg_elig) elig = p.elig[u.bh] != 0;
    for (int k = 0; elig && p.seg_elig && k < g[0]; ++k)
        elig = p.seg_elig[(size_t)u.bh * p.nseg + g[kGatherPiece + 3 * k]] != 0;
    u.stat = p.mode == VDIT_MODE_FORCE_STATIC || elig;
    u.alt = u.nkt >= 2;
}

// Row r of gathered tile `gat`: its sequence row, and in seg its segment. Rows
// past the last piece repeat that piece's rows (computed, never stored).
__device__ __forceinline__ int gathered_row(const Params &p, int gat, int r, int &seg) {
    const int32_t *g = p.gathers + kGatherInts * gat;
    int k = 0, off = 0;
    while (k < g[0] - 1 && r >= off + g[kGatherPiece + 3 * k + 2]) {
        off += g[kGatherPiece + 3 * k + 2];
        ++k;
    }
    seg = g[kGatherPiece + 3 * k];
    return g[kGatherPiece + 3 * k + 1] + (r - off) % g[kGatherPiece + 3 * k + 2];
}

template <int kMode>
__device__ __forceinline__ void decode_any(const Params &p, long long w, Work &u) {
    if constexpr (kMode == kModeTiled) decode_tiled(p, w, u);
    else if constexpr (kMode == kModeGathered) decode_gathered(p, w, u);
    else decode(p, w, u);
}

// Live key runs of query row i under the frame-blind tiling (the padded tail
// takes the last frame's): [lo0, hi0) and [lo1, hi1), possibly empty.
__device__ __forceinline__ void row_runs(const Params &p, int i, int &lo0, int &hi0, int &lo1, int &hi1) {
    const int f = min(i, p.N - 1) / p.T;
    const int wlo = max(0, f - p.W), whi = min(p.F - 1, f + p.W);
    const bool ref_out = p.ref >= 0 && (p.ref < wlo || p.ref > whi);
    lo0 = hi0 = lo1 = hi1 = 0;
    if (p.part != VDIT_PART_REFERENCE) { lo0 = wlo * p.T; hi0 = (whi + 1) * p.T; }
    if (p.part != VDIT_PART_WINDOW && ref_out) { lo1 = p.ref * p.T; hi1 = (p.ref + 1) * p.T; }
}

// first row of query tile q of the unit (last tile of a segment ends at its end)
__device__ __forceinline__ int tile_row(const Work &u, int q) {
    const int t = kTilesPerUnit * u.pair + q;
    const int off = min(t * kTileRows, max(u.rows - kTileRows, 0));
    return u.row0 + off;
}

// key tile j: first key and number of live keys
__device__ __forceinline__ void key_tile(const Work &u, int j, int &start, int &nvalid) {
    if (j < u.nt0) {
        start = u.lo0 + j * kBK;
        nvalid = min(kBK, u.hi0 - start);
    } else {
        start = u.lo1 + (j - u.nt0) * kBK;
        nvalid = min(kBK, u.hi1 - start);
    }
}

// Wait that ignores the abort flag, used only to drain in-flight copies/MMAs
// before exit. It always allows the default limit (not the possibly shortened
// limit of the ordinary waits): copies and MMAs already issued must land
// before the CTA's shared memory and TMEM are released.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) return false;
    }
    return true;
}

// tm_q: 128-row boxes; in the gathered instance 16-row boxes (pieces are
// multiples of 16 rows)
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const Params p) {
    constexpr bool kTiled = kMode == kModeTiled;
    constexpr bool kGathered = kMode == kModeGathered;
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + L::kBar;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kBar + 8 * kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kBar + 8 * kNumBars + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint64_t tlim = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQfull), 1);
        mbar_init(bar(kBarQfree), 1 + 8);
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(bar(kBarKfull + s), 1);
            mbar_init(bar(kBarKfree + s), 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(bar(kBarVfull + s), 1);
            mbar_init(bar(kBarVfree + s), 1);
        }
        for (int q = 0; q < kTilesPerUnit; ++q) {
            mbar_init(bar(kBarSfull + q), 1);
            mbar_init(bar(kBarPfull + q), 4);
            mbar_init(bar(kBarOfull + q), 1);
            mbar_init(bar(kBarOfree + q), 4);
        }
        mbar_init(bar(kBarFinal), 1);
        mbar_init(bar(kBarXfull), 4);   // row sums of slot 1, passed to warpgroup 0
        mbar_init(bar(kBarXfree), 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the gathered-tile launch that follows may place its CTAs as SMs free up
    if constexpr (kMode == kModeAligned) grid_launch_dependents();

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t nk = 0, nv = 0, it = 0;  // K tiles, V tiles and Q pairs issued
            bool ok = true;
            for (long long w = blockIdx.x; ok && w < p.total_work; w += gridDim.x) {
                Work u;
                decode_any<kMode>(p, w, u);
                if (kTiled && u.nkt == 0) continue;   // a block with no live key: no work
                if (!(ok = mbar_wait(bar(kBarQfree), (it & 1) ^ 1, abort_flag, p.status, kSiteQfree, tlim)))
                    break;
                mbar_arrive_expect_tx(bar(kBarQfull), (uint32_t)(u.nact * L::kTileBytes));
                if constexpr (kGathered) {
                    // 16-row groups from the tile's pieces
                    for (int r0 = 0; r0 < kTileRows; r0 += 16) {
                        int sg;
                        const int row = gathered_row(p, u.gat, r0, sg);
                        for (int hf = 0; hf < D / 64; ++hf)
                            tma_load_4d(sbase + L::kQ + hf * kHalfBytes + r0 * 128, &tm_q, bar(kBarQfull),
                                        hf * 64, row, u.h, u.b);
                    }
                } else {
                    for (int q = 0; q < u.nact; ++q) {
                        const int row = tile_row(u, q);
                        for (int hf = 0; hf < D / 64; ++hf)
                            tma_load_4d(sbase + L::kQ + q * L::kTileBytes + hf * kHalfBytes, &tm_q,
                                        bar(kBarQfull), hf * 64, row, u.h, u.b);
                    }
                }
                ++it;
                for (int j = 0; j < u.nkt; ++j) {
                    int start, nvalid;
                    key_tile(u, j, start, nvalid);
                    const int sk = nk % kStagesK;
                    if (!(ok = mbar_wait(bar(kBarKfree + sk), ((nk / kStagesK) & 1) ^ 1, abort_flag,
                                         p.status, kSiteKfree, tlim)))
                        break;
                    mbar_arrive_expect_tx(bar(kBarKfull + sk), L::kTileBytes);
                    for (int hf = 0; hf < D / 64; ++hf)
                        tma_load_4d(sbase + L::kK + sk * L::kTileBytes + hf * kHalfBytes, &tm_k,
                                    bar(kBarKfull + sk), hf * 64, start, u.h, u.b);
                    ++nk;
                    const int sv = nv % kStagesV;
                    if (!(ok = mbar_wait(bar(kBarVfree + sv), ((nv / kStagesV) & 1) ^ 1, abort_flag,
                                         p.status, kSiteVfree, tlim)))
                        break;
                    mbar_arrive_expect_tx(bar(kBarVfull + sv), L::kTileBytes);
                    for (int hf = 0; hf < D / 64; ++hf)
                        tma_load_4d(sbase + L::kV + sv * L::kTileBytes + hf * kHalfBytes, &tm_v,
                                    bar(kBarVfull + sv), hf * 64, start, u.h, u.b);
                    ++nv;
                }
            }
            // drain: every copy this thread issued must land before the CTA exits
            for (int s = 0; s < kStagesK; ++s) {
                const uint32_t n_k = nk / kStagesK + ((uint32_t)s < nk % kStagesK ? 1u : 0u);
                if (n_k > 0) drain_wait(bar(kBarKfull + s), (n_k - 1) & 1, kDefaultTimeoutNs);
            }
            for (int s = 0; s < kStagesV; ++s) {
                const uint32_t n_v = nv / kStagesV + ((uint32_t)s < nv % kStagesV ? 1u : 0u);
                if (n_v > 0) drain_wait(bar(kBarVfull + s), (n_v - 1) & 1, kDefaultTimeoutNs);
            }
            if (it > 0) drain_wait(bar(kBarQfull), (it - 1) & 1, kDefaultTimeoutNs);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the schedule (warp-uniform control flow) and one
        // elected lane issues every tcgen05.mma and commit. A tcgen05.mma issue
        // returns only when the tensor pipe can take it, so anything computed
        // between two MMAs is idle tensor time: descriptors are built once and
        // K-steps add compile-time offsets to the start-address field.
        const bool leader = elect_one();
        constexpr uint32_t kTileDesc = L::kTileBytes >> 4;   // one tile, in descriptor address units
        const uint64_t dQ = sdesc_sw128(sbase + L::kQ, 16, 1024);
        const uint64_t dK = sdesc_sw128(sbase + L::kK, 16, 1024);
        const uint64_t dV = sdesc_sw128(sbase + L::kV, kHalfBytes, 1024);
        const uint32_t tS0 = tmem + L::kTmemS, tO0 = tmem + L::kTmemO;
        constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
        constexpr uint32_t kIdescS = idesc_bf16(128, kBK, false);
        // S_q = Q_q K^T (K-major A and B); a tail tile uses a narrower N
        auto issue_s = [&](int q, int sk, int nmma, int qt) {   // slot q, Q tile qt
            const uint64_t a0 = dQ + (uint64_t)(qt * kTileDesc);
            const uint64_t b0 = dK + (uint64_t)(sk * kTileDesc);
            const uint32_t idesc = nmma == kBK ? kIdescS : idesc_bf16(128, nmma, false);
            const uint32_t d = tS0 + q * 128;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks / 4) * (kHalfBytes >> 4) + (ks % 4) * 2;
                mma_ss(d, a0 + off, b0 + off, idesc, ks > 0 ? 1u : 0u);
            }
        };
        // O_q (+)= P_q V: P from TMEM (8 packed columns per 16 keys), V MN-major
        auto issue_pv = [&](int q, int sv, int nmma, bool acc) {
            const uint64_t b0 = dV + (uint64_t)(sv * kTileDesc);
            const uint32_t d = tO0 + q * D, a = tS0 + q * 128;
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks) {
                if (ks * 16 < nmma)
                    mma_ts(d, a + ks * 8, b0 + ks * (2048 >> 4), kIdescPV, (ks > 0 || acc) ? 1u : 0u);
            }
        };
        auto wait = [&](int b, uint32_t parity, int site) {
            return mbar_wait_warp(bar(b), parity, abort_flag, p.status, site, tlim);
        };
        uint32_t kc = 0, it = 0, sq[kTilesPerUnit] = {0, 0}, uq[kTilesPerUnit] = {0, 0};
        bool ok = true;
        for (long long w = blockIdx.x; ok && w < p.total_work; w += gridDim.x, ++it) {
            Work u;
            decode_any<kMode>(p, w, u);
            if (kTiled && u.nkt == 0) { --it; continue; }   // skipped by every role: no phase used
            if (!(ok = wait(kBarQfull, it & 1, kSiteQfullMma))) break;
            const uint32_t kc0 = kc;
            int start, nvalid;
            if (u.alt) {
                // slot j % 2 takes key tile j: S of key tiles 0 and 1, then per key
                // tile j its P.V and the S of key tile j + 2 into the same slot
#pragma unroll
                for (int q = 0; q < kTilesPerUnit; ++q) {
                    const uint32_t c = kc0 + q;
                    const int sk = c % kStagesK;
                    key_tile(u, q, start, nvalid);
                    if (!(ok = wait(kBarKfull + sk, (c / kStagesK) & 1, kSiteKfull))) break;
                    tc_fence_after();
                    if (leader) {
                        issue_s(q, sk, (nvalid + 15) & ~15, 0);
                        mma_commit(bar(kBarSfull + q));
                    }
                    __syncwarp();
                }
                for (int j = 0; j < u.nkt && ok; ++j) {
                    const int q = j & 1;
                    const uint32_t c = kc0 + j;
                    const int sv = c % kStagesV;
                    key_tile(u, j, start, nvalid);
                    const int nmma = (nvalid + 15) & ~15;
                    if (!(ok = wait(kBarVfull + sv, (c / kStagesV) & 1, kSiteVfull))) break;
                    if (!(ok = wait(kBarPfull + q, sq[q] & 1, kSitePfull))) break;
                    if (j == q && !(ok = wait(kBarOfree + q, (uq[q] & 1) ^ 1, kSiteOfree))) break;
                    tc_fence_after();
                    if (leader) {
                        issue_pv(q, sv, nmma, j >= 2);
                        if (j + 2 >= u.nkt) mma_commit(bar(kBarOfull + q));
                    }
                    ++sq[q];
                    if (j + 2 < u.nkt) {
                        const uint32_t c2 = c + 2;
                        const int sk2 = c2 % kStagesK;
                        int start2, nvalid2;
                        key_tile(u, j + 2, start2, nvalid2);
                        if (!(ok = wait(kBarKfull + sk2, (c2 / kStagesK) & 1, kSiteKfull))) break;
                        tc_fence_after();
                        if (leader) {
                            issue_s(q, sk2, (nvalid2 + 15) & ~15, 0);
                            mma_commit(bar(kBarSfull + q));
                        }
                    }
                    __syncwarp();
                }
                ++uq[0];
                ++uq[1];
                kc += u.nkt;
                continue;
            }
            key_tile(u, 0, start, nvalid);

            {
                const int sk = kc0 % kStagesK;
                if (!(ok = wait(kBarKfull + sk, (kc0 / kStagesK) & 1, kSiteKfull))) break;
                tc_fence_after();
                if (leader) {
                    for (int q = 0; q < u.nact; ++q) {
                        issue_s(q, sk, (nvalid + 15) & ~15, q);
                        mma_commit(bar(kBarSfull + q));
                    }
                }
            }
            for (int j = 0; j < u.nkt && ok; ++j) {
                const uint32_t c = kc0 + j;
                const int sv = c % kStagesV;
                key_tile(u, j, start, nvalid);
                const int nmma = (nvalid + 15) & ~15;
                int start1 = 0, nvalid1 = 0;
                if (j + 1 < u.nkt) key_tile(u, j + 1, start1, nvalid1);
                const uint32_t c1 = c + 1;
                const int sk1 = c1 % kStagesK;
                if (!(ok = wait(kBarVfull + sv, (c / kStagesV) & 1, kSiteVfull))) break;
                for (int q = 0; q < u.nact && ok; ++q) {
                    if (!(ok = wait(kBarPfull + q, sq[q] & 1, kSitePfull))) break;
                    if (j == 0 && !(ok = wait(kBarOfree + q, (uq[q] & 1) ^ 1, kSiteOfree))) break;
                    tc_fence_after();
                    if (leader) {
                        issue_pv(q, sv, nmma, j > 0);
                        if (j == u.nkt - 1) mma_commit(bar(kBarOfull + q));
                    }
                    ++sq[q];
                    if (j + 1 < u.nkt) {
                        if (q == 0) {
                            if (!(ok = wait(kBarKfull + sk1, (c1 / kStagesK) & 1, kSiteKfull))) break;
                            tc_fence_after();
                        }
                        if (leader) {
                            issue_s(q, sk1, (nvalid1 + 15) & ~15, q);
                            mma_commit(bar(kBarSfull + q));
                        }
                    }
                }
            }
            for (int q = 0; q < u.nact; ++q) ++uq[q];
            kc += u.nkt;
        }
        // drain: all issued MMAs complete before TMEM is released
        if (leader) mma_commit(bar(kBarFinal));
        __syncwarp();
        drain_wait(bar(kBarFinal), 0, kDefaultTimeoutNs);
    } else if (warp >= kWarpSoftmax0) {
        // ------------------------------------------------------------ softmax warpgroups
        const int q = (warp - kWarpSoftmax0) / 4; // query tile of this warpgroup
        const int r = threadIdx.x % kTileRows;   // row within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp % 4)) << 16;
        const uint32_t tS = tmem + L::kTmemS + q * 128 + lane_off;
        const uint32_t tO = tmem + L::kTmemO + q * D + lane_off;
        const uint32_t tO1 = tmem + L::kTmemO + D + lane_off;     // slot 1's O (alternating units)
        const float sc = p.scale_log2;
        float *xbuf = reinterpret_cast<float *>(smem + L::kX);
        // uq: own slot's O-ready phases; uo1 (warpgroup 0): slot 1's; xc: row-sum handovers
        uint32_t it = 0, sq = 0, uq = 0, kc = 0, uo1 = 0, xc = 0;
        bool ok = true;
        for (long long w = blockIdx.x; ok && w < p.total_work; w += gridDim.x, ++it) {
            Work u;
            decode_any<kMode>(p, w, u);
            if (kTiled && u.nkt == 0) {
                // skipped by every role (no phase used): a block none of whose rows
                // sees a key of this part of the mask stores O = 0 and LSE = -inf
                const int row = tile_row(u, q) + r;
                if (q < u.nact && row < p.N) {
                    const long long obase = (long long)u.b * p.os0 + (long long)u.h * p.os1 + (long long)row * p.os2;
                    for (int c0 = 0; c0 < D; c0 += 8) {
                        if (p.o_f32) {
                            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.o) + obase + c0);
                            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                        } else {
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + obase + c0) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    if (p.lse) p.lse[((long long)u.bh * p.N) + row] = -INFINITY;
                }
                --it;
                continue;
            }
            const bool act = q < u.nact || u.alt;
            // The last active warpgroup releases K, V and Q tiles: its S barrier for key
            // tile j is committed after every earlier MMA of the unit (all S MMAs of
            // tile j, all P.V MMAs of tile j-1); its O barrier covers the last P.V.
            const bool releaser = !u.alt && q == u.nact - 1 && (warp % 4) == 0 && lane == 0;
            // alternating units: each warpgroup releases the K (and V two key tiles
            // back) of its own key tiles
            const bool rel_alt = u.alt && (warp % 4) == 0 && lane == 0;
            const uint32_t kc0 = kc;
            kc += u.nkt;
            const bool stat = u.stat;
            ok = mbar_wait_warp(bar(kBarQfull), it & 1, abort_flag, p.status, kSiteQfullSm, tlim);
            if (!ok) break;
            // a gathered tile's row: its segment (the bound's R, the row's key runs)
            int gseg = u.seg;
            if constexpr (kGathered) gathered_row(p, u.gat, r, gseg);
            // row bound ("Unchaining the Softmax"): m~ = scale*log2e*(q.c + |q| R)
            float mt = 0.f;
            if (act && stat) {
                const uint8_t *qt = smem + L::kQ + (u.alt ? 0 : q) * L::kTileBytes;
                const float *cm = p.k_mean + (size_t)u.bh * D;
                float dot = 0.f, nn = 0.f;
#pragma unroll
                for (int hf = 0; hf < D / 64; ++hf) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            qt + hf * kHalfBytes + r * 128 + ((ch ^ (r & 7)) * 16));
                        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = __uint_as_float(wv[e] << 16);
                            const float x1 = __uint_as_float(wv[e] & 0xFFFF0000u);
                            const int d = hf * 64 + ch * 8 + 2 * e;
                            dot = fmaf(x0, cm[d], dot);
                            dot = fmaf(x1, cm[d + 1], dot);
                            nn = fmaf(x0, x0, nn);
                            nn = fmaf(x1, x1, nn);
                        }
                    }
                }
                const float R = p.seg_rmax ? p.seg_rmax[(size_t)u.bh * p.nseg + gseg] : p.k_rmax[u.bh];
                mt = sc * (dot + sqrtf(nn) * R);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarQfree));
            if (!act) continue;

            float l0 = 0.f, l1 = 0.f, mrun = -INFINITY;
            const int j0 = u.alt ? q : 0;          // this warpgroup's first key tile
            int rlo0 = 0, rhi0 = 0, rlo1 = 0, rhi1 = 0;   // this row's live keys
            if constexpr (kTiled) row_runs(p, tile_row(u, u.alt ? 0 : q) + r, rlo0, rhi0, rlo1, rhi1);
            if constexpr (kGathered) {
                const int32_t *sg = p.segments + kSegInts * gseg;
                rlo0 = sg[2]; rhi0 = sg[3]; rlo1 = sg[4]; rhi1 = sg[5];
            }
            for (int j = j0; j < u.nkt; j += u.alt ? 2 : 1) {
                int start, nvalid;
                key_tile(u, j, start, nvalid);
                ok = mbar_wait_warp(bar(kBarSfull + q), sq & 1, abort_flag, p.status, kSiteSfull, tlim);
                if (!ok) break;
                tc_fence_after();
                if (releaser) {
                    mbar_arrive(bar(kBarKfree + (kc0 + j) % kStagesK));
                    if (j > 0) mbar_arrive(bar(kBarVfree + (kc0 + j - 1) % kStagesV));
                    if (j == u.nkt - 1) mbar_arrive(bar(kBarQfree));
                }
                if (rel_alt) {
                    // S_q(j) was issued after P_q(j-2).V: K_j and V_{j-2} are free;
                    // the last key tile's S is the unit's last S: Q is free
                    mbar_arrive(bar(kBarKfree + (kc0 + j) % kStagesK));
                    if (j >= 2) mbar_arrive(bar(kBarVfree + (kc0 + j - 2) % kStagesV));
                    if (j == u.nkt - 1) mbar_arrive(bar(kBarQfree));
                }
                // p = 2^(s*scale*log2e - mrow), P -> bf16 into the first half of S, from
                // the 128-column S row in registers
                auto exps = [&](uint32_t (&v)[128], float mrow) {
                    const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(-mrow, -mrow);
                    uint64_t l2 = f2_pack(0.f, 0.f);
                    // all 64 packed P columns first, then one TMEM store (measured faster
                    // than storing each 32-column half as soon as it is ready)
                    uint32_t pk[64];
                    if (nvalid >= kBK) {
                        // column pairs: one f32x2 FMA for the scaled, shifted logits and one
                        // f32x2 add for the row sums
                        static_for<64>([&](auto E) {
                            constexpr int e = decltype(E)::value;
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc2, nm2),
                                      x0, x1);
                            const float p0 = ex2(x0);
                            const float p1 = ex2(x1);
                            l2 = f2_add(l2, f2_pack(p0, p1));
                            pk[e] = pack_bf16(p0, p1);
                        });
                    } else {
#pragma unroll
                        for (int e = 0; e < 64; ++e) {
                            const int i0 = 2 * e;
                            const float p0 = i0 < nvalid ? ex2(fmaf(__uint_as_float(v[i0]), sc, -mrow)) : 0.f;
                            const float p1 = i0 + 1 < nvalid ? ex2(fmaf(__uint_as_float(v[i0 + 1]), sc, -mrow)) : 0.f;
                            l0 += p0;
                            l1 += p1;
                            pk[e] = pack_bf16(p0, p1);
                        }
                    }
                    tmem_st64(tS, pk);
                    float a0, a1;
                    f2_unpack(l2, a0, a1);
                    l0 += a0;
                    l1 += a1;
                };
                // frame-blind tiling: in a tile that straddles a frame boundary the mask
                // predicate, per element, turns this row's dead keys (and padding) into
                // -inf. Gathered tiles mask each row to its own key runs; there a row
                // that sees no key of the tile returns true and takes an infinite shift
                // (p = 0) instead, unless the warp masks per element anyway because one
                // of its rows straddles a run boundary.
                auto mask = [&](uint32_t (&v)[128]) -> bool {
                    if constexpr (kTiled || kGathered) {
                        const int kend = start + (kTiled ? kBK : nvalid);
                        const bool full = (rlo0 <= start && kend <= rhi0) || (rlo1 <= start && kend <= rhi1);
                        const bool dead =
                            kGathered && !(rlo0 < kend && start < rhi0) && !(rlo1 < kend && start < rhi1);
                        if (!__all_sync(0xffffffffu, full || dead)) {
#pragma unroll
                            for (int e = 0; e < 128; ++e) {
                                const int jk = start + e;
                                const bool live = (unsigned)(jk - rlo0) < (unsigned)(rhi0 - rlo0) ||
                                                  (unsigned)(jk - rlo1) < (unsigned)(rhi1 - rlo1);
                                v[e] = live ? v[e] : 0xff800000u;
                            }
                            return false;
                        }
                        return dead;
                    }
                    return false;
                };
                // Each path loads the whole S row in one TMEM load of its own: a load
                // shared by both paths ahead of the branch measured 8% slower on the
                // static path.
                if (stat) {
                    uint32_t v[128];
                    tmem_ld128(tS, v);
                    const bool dead = mask(v);
                    exps(v, dead ? INFINITY : mt);
                } else {
                    uint32_t v[128];
                    tmem_ld128(tS, v);
                    const bool dead = mask(v);
                    // online: this tile's row max, taken on the raw logits (the scale is
                    // positive), then the lazy rescale decision
                    float mx;
                    if (nvalid >= kBK) {
                        float m8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) m8[e] = __uint_as_float(v[e]);
#pragma unroll
                        for (int e = 8; e < 128; ++e) m8[e % 8] = fmaxf(m8[e % 8], __uint_as_float(v[e]));
                        mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                    } else {
                        mx = -INFINITY;
#pragma unroll
                        for (int e = 0; e < 128; ++e) mx = e < nvalid ? fmaxf(mx, __uint_as_float(v[e])) : mx;
                    }
                    mx = dead ? -INFINITY : mx * sc;
                    float alpha = 1.f;      // factor of the O rescale (lazy, warp-uniform)
                    bool rescale = false;
                    if (j == j0) {
                        mrun = mx;
                    } else {
                        const bool need = mx > mrun + kLazyRescale;
                        if (__any_sync(0xffffffffu, need)) {
                            rescale = true;
                            alpha = need ? ex2(mrun - mx) : 1.f;
                            l0 *= alpha;
                            l1 *= alpha;
                            if (need) mrun = mx;
                        }
                    }
                    // no live key in this row yet (frame-blind tiling, gathered tile):
                    // every term is masked, any finite shift gives p = 0
                    exps(v, dead ? INFINITY : ((kTiled || kGathered) && mrun == -INFINITY ? 0.f : mrun));
                    if (rescale) {
                        // O (after P.V of the previous key tile, which the S barrier of
                        // this tile covers) scaled to the new running max, before this
                        // tile's P.V
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32(tO + c0, o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + c0, o);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarPfull + q));
                ++sq;
                if (!stat) mt = mrun;
            }
            if (!ok) break;
            float l = l0 + l1;
            float w0 = 1.f, w1 = 1.f;   // weights of O0 and O1 in an alternating online unit
            if (u.alt) {
                // warpgroup 1 hands its row sums (and, online, its running max) to
                // warpgroup 0, which writes the tile
                if (q == 1) {
                    ok = mbar_wait_warp(bar(kBarXfree), (xc & 1) ^ 1, abort_flag, p.status, kSiteXfree, tlim);
                    if (!ok) break;
                    xbuf[r] = l;
                    xbuf[kTileRows + r] = mt;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kBarXfull));
                    ++xc;
                    ++uq;
                    continue;
                }
                ok = mbar_wait_warp(bar(kBarXfull), xc & 1, abort_flag, p.status, kSiteXfull, tlim);
                if (!ok) break;
                if (stat) {
                    l += xbuf[r];       // both halves share the static bound
                } else {
                    // online halves have their own running maxima m0, m1: rescale both
                    // to M = max(m0, m1), which is exact (softmax is shift-invariant)
                    const float m1 = xbuf[kTileRows + r], M = fmaxf(mt, m1);
                    w0 = ex2(mt - M);
                    w1 = ex2(m1 - M);
                    if constexpr (kTiled) {
                        // a half that saw no live key has l = 0 and takes no weight
                        w0 = mt == -INFINITY ? 0.f : w0;
                        w1 = m1 == -INFINITY ? 0.f : w1;
                    }
                    l = l * w0 + xbuf[r] * w1;
                    mt = M;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarXfree));
                ++xc;
                ok = mbar_wait_warp(bar(kBarOfull + 1), uo1 & 1, abort_flag, p.status, kSiteOfull, tlim);
                if (!ok) break;
            }
            ok = mbar_wait_warp(bar(kBarOfull + q), uq & 1, abort_flag, p.status, kSiteOfull, tlim);
            if (!ok) break;
            tc_fence_after();
            if (releaser) mbar_arrive(bar(kBarVfree + (kc0 + u.nkt - 1) % kStagesV));
            if (rel_alt) {
                mbar_arrive(bar(kBarVfree + (kc0 + u.nkt - 2) % kStagesV));
                mbar_arrive(bar(kBarVfree + (kc0 + u.nkt - 1) % kStagesV));
            }
            // epilogue: O / l for the rows this tile owns, and LSE (alternating
            // units: O = O0 + O1, online O = w0 O0 + w1 O1)
            // a row that saw no live key at all (possible only for a part of the
            // mask under the frame-blind tiling) stores O = 0 and LSE = -inf
            const float inv = kTiled && l == 0.f ? 0.f : 1.0f / l;
            const int t = kTilesPerUnit * u.pair + q;
            const int row = kGathered ? gathered_row(p, u.gat, r, gseg) : tile_row(u, q) + r;
            const int own_lo = u.row0 + t * kTileRows;
            const int own_hi = u.row0 + min((t + 1) * kTileRows, u.rows);
            const bool owned = kGathered ? r < u.rows : row >= own_lo && row < own_hi && (!kTiled || row < p.N);
            const long long obase = (long long)u.b * p.os0 + (long long)u.h * p.os1 + (long long)row * p.os2;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tO + c0, v);
                if (u.alt) {
                    uint32_t v1[32];
                    tmem_ld32(tO1 + c0, v1);
                    if (stat) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(v1[e]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(fmaf(__uint_as_float(v[e]), w0, __uint_as_float(v1[e]) * w1));
                    }
                }
                if (owned) {
                    if (p.o_f32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.o) + obase + c0);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(v[4 * e]) * inv,
                                                 __uint_as_float(v[4 * e + 1]) * inv,
                                                 __uint_as_float(v[4 * e + 2]) * inv,
                                                 __uint_as_float(v[4 * e + 3]) * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + obase + c0);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint4 o4;
                            o4.x = pack_bf16(__uint_as_float(v[8 * e + 0]) * inv, __uint_as_float(v[8 * e + 1]) * inv);
                            o4.y = pack_bf16(__uint_as_float(v[8 * e + 2]) * inv, __uint_as_float(v[8 * e + 3]) * inv);
                            o4.z = pack_bf16(__uint_as_float(v[8 * e + 4]) * inv, __uint_as_float(v[8 * e + 5]) * inv);
                            o4.w = pack_bf16(__uint_as_float(v[8 * e + 6]) * inv, __uint_as_float(v[8 * e + 7]) * inv);
                            dst[e] = o4;
                        }
                    }
                }
            }
            if (owned && p.lse)
                p.lse[((long long)u.bh * p.N) + row] = (mt + log2f(l)) * 0.69314718055994531f;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(kBarOfree + q));
                if (u.alt) mbar_arrive(bar(kBarOfree + 1));
            }
            ++uq;
            if (q == 0 && (u.nact == 2 || u.alt)) ++uo1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // the gathered launch completes only after the launch it depends on, so work
    // the stream orders after it also follows that launch
    if constexpr (kGathered) grid_dependency_wait();
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [B, H, N, D] bf16 tensor -> 4-D tensor map with a 64 x rows x 1 x 1 box, 128-byte swizzle.
bool encode_bhnd(CUtensorMap *m, const void *base, int B, int H, int N, int D, const int64_t st[3],
                 unsigned rows = 128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
    cuuint32_t box[4] = {64, rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Both head dims request the D = 128 shared-memory size: one CTA (and so one
// TMEM owner) per SM.
constexpr int kSmemRequest = Layout<128>::kAlloc;   // both head dims launch with this size
static_assert(Layout<64>::kBytes <= Layout<64>::kAlloc && Layout<64>::kAlloc <= kSmemRequest,
              "the D = 64 layout must fit the shared-memory request");
static_assert(kSmemRequest <= 227 * 1024, "shared memory beyond the per-CTA limit");

template <int D, int kMode>
cudaError_t prepare_kernel(int device) {
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> g(mu);
    if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemRequest);
    if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
    return e;
}

// Merge of two partial attention results over disjoint key sets (the window
// pass a and the reference pass b of the two-pass form): per row, with
// M = max(LSE_a, LSE_b), w_x = exp(LSE_x - M),
//   O = (w_a O_a + w_b O_b) / (w_a + w_b),   LSE = M + ln(w_a + w_b).
// Rows whose frame has no key in plan b take pass a unchanged. One warp per
// row; O_a, O_b fp32 [BH, N, D] and LSE_a, LSE_b fp32 [BH, N], dense.
__global__ void merge_kernel(const float *oa, const float *la, const float *ob, const float *lb,
                             const int32_t *runs_b, int T, int N, int H, long long rows, int D,
                             void *o, long long os0, long long os1, long long os2, int o_f32,
                             float *lse) {
    const int lane = threadIdx.x % 32;
    const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
    for (long long rw = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32; rw < rows; rw += nwarps) {
        const int bh = (int)(rw / N), i = (int)(rw % N), f = i / T;
        const int32_t *rb = runs_b + 4 * f;
        const bool has_b = rb[1] > rb[0] || rb[3] > rb[2];
        const float lsa = la[rw];
        float wa = 1.f, wb = 0.f, L = lsa;
        if (has_b) {
            const float lsb = lb[rw], M = fmaxf(lsa, lsb);
            wa = expf(lsa - M);
            wb = expf(lsb - M);
            const float sum = wa + wb;
            wa /= sum;
            wb /= sum;
            L = M + logf(sum);
        }
        const long long obase = (long long)(bh / H) * os0 + (long long)(bh % H) * os1 + (long long)i * os2;
        for (int c = lane * 4; c < D; c += 128) {
            const float4 a = *reinterpret_cast<const float4 *>(oa + rw * D + c);
            float4 r = make_float4(a.x * wa, a.y * wa, a.z * wa, a.w * wa);
            if (has_b) {
                const float4 b = *reinterpret_cast<const float4 *>(ob + rw * D + c);
                r = make_float4(fmaf(b.x, wb, r.x), fmaf(b.y, wb, r.y), fmaf(b.z, wb, r.z), fmaf(b.w, wb, r.w));
            }
            if (o_f32) {
                *reinterpret_cast<float4 *>(static_cast<float *>(o) + obase + c) = r;
            } else {
                uint2 pk;
                pk.x = pack_bf16(r.x, r.y);
                pk.y = pack_bf16(r.z, r.w);
                *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(o) + obase + c) = pk;
            }
        }
        if (lse && lane == 0) lse[rw] = L;
    }
}

int sm_count(int device) {
    static std::mutex mu;
    static int cache[64] = {};
    std::lock_guard<std::mutex> g(mu);
    if (device < 0 || device >= 64) return 0;
    if (cache[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) == cudaSuccess)
            cache[device] = n;
    }
    return cache[device];
}

}  // namespace
}  // namespace vdit

using namespace vdit;

namespace {
vdit_status attn_fwd_impl(const vdit_plan *plan, const void *q, const void *k, const void *v, void *o,
                          int32_t o_dtype, float *lse, int32_t B, int32_t H, int32_t D,
                          const int64_t q_strides[3], const int64_t k_strides[3],
                          const int64_t v_strides[3], const int64_t o_strides[3], float scale,
                          const float *k_mean, const float *k_rmax, const uint8_t *eligible,
                          const float *seg_rmax, const uint8_t *seg_elig, int32_t mode,
                          void *stream, bool tiled = false) {
    clear_error();
    if (!plan) { set_error("vdit_attn_fwd: plan is NULL"); return VDIT_ERR_INVALID; }
    if (!q || !k || !v || !o || !q_strides || !k_strides || !v_strides || !o_strides) {
        set_error("vdit_attn_fwd: NULL tensor or stride argument");
        return VDIT_ERR_INVALID;
    }
    if (B < 1 || H < 1) { set_error("vdit_attn_fwd: B=%d H=%d must be >= 1", B, H); return VDIT_ERR_INVALID; }
    if (D != 64 && D != 128) {
        set_error("vdit_attn_fwd: head dim D=%d not supported (64 or 128)", D);
        return VDIT_ERR_UNSUPPORTED;
    }
    if (o_dtype != VDIT_O_BF16 && o_dtype != VDIT_O_F32) {
        set_error("vdit_attn_fwd: o_dtype=%d invalid", o_dtype);
        return VDIT_ERR_INVALID;
    }
    if (mode < VDIT_MODE_AUTO || mode > VDIT_MODE_FORCE_STATIC) {
        set_error("vdit_attn_fwd: mode=%d invalid", mode);
        return VDIT_ERR_INVALID;
    }
    if (mode != VDIT_MODE_FORCE_ONLINE && (!k_mean || !k_rmax)) {
        set_error("vdit_attn_fwd: k_mean and k_rmax are required unless mode is FORCE_ONLINE");
        return VDIT_ERR_INVALID;
    }
    if (mode == VDIT_MODE_AUTO && !eligible) {
        set_error("vdit_attn_fwd: eligible is required in AUTO mode");
        return VDIT_ERR_INVALID;
    }
    if (!finite_positive(scale)) { set_error("vdit_attn_fwd: scale must be finite and > 0"); return VDIT_ERR_INVALID; }
    const int64_t *sts[3] = {q_strides, k_strides, v_strides};
    for (int t = 0; t < 3; ++t)
        for (int i = 0; i < 3; ++i)
            if (sts[t][i] <= 0 || sts[t][i] % 8 != 0 || sts[t][i] >= (1ll << 38)) {
                set_error("vdit_attn_fwd: q/k/v strides must be positive multiples of 8 elements");
                return VDIT_ERR_INVALID;
            }
    const int oal = o_dtype == VDIT_O_F32 ? 4 : 8;
    for (int i = 0; i < 3; ++i)
        if (o_strides[i] <= 0 || o_strides[i] % oal != 0) {
            set_error("vdit_attn_fwd: o strides must be positive multiples of 16 bytes");
            return VDIT_ERR_INVALID;
        }
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) {
        set_error("vdit_attn_fwd: q, k, v, o must be 16-byte aligned");
        return VDIT_ERR_INVALID;
    }
    int dev = -1;
    VDIT_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != plan->device) {
        set_error("vdit_attn_fwd: plan was built on device %d, current device is %d", plan->device, dev);
        return VDIT_ERR_INVALID;
    }
    const int N = (int)plan->N;
    // the gathered tiles (second launch) read Q in 16-row boxes
    const bool gathered = !tiled && plan->h.n_gathers > 0;
    CUtensorMap tq, tk, tv, tq16;
    if (!encode_bhnd(&tq, q, B, H, N, D, q_strides) || !encode_bhnd(&tk, k, B, H, N, D, k_strides) ||
        !encode_bhnd(&tv, v, B, H, N, D, v_strides) || (gathered && !encode_bhnd(&tq16, q, B, H, N, D, q_strides, 16))) {
        set_error("vdit_attn_fwd: cuTensorMapEncodeTiled failed (alignment/strides or driver entry point)");
        return VDIT_ERR_INVALID;
    }
    Params prm;
    prm.segments = plan->d_segments;
    prm.units = plan->d_units;
    prm.class_off = plan->d_class_off;
    prm.n_classes = plan->h.n_classes;
    prm.B = B; prm.H = H; prm.N = N;
    prm.total_work = (long long)B * H * plan->h.n_units;
    prm.o = o;
    prm.os0 = o_strides[0]; prm.os1 = o_strides[1]; prm.os2 = o_strides[2];
    prm.o_f32 = o_dtype == VDIT_O_F32;
    prm.lse = lse;
    prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
    prm.k_mean = k_mean; prm.k_rmax = k_rmax; prm.elig = eligible;
    prm.seg_rmax = seg_rmax; prm.seg_elig = seg_elig; prm.nseg = plan->h.n_segments;
    prm.mode = mode;
    prm.status = plan->d_status;
    prm.timeout_ns = wait_limit_ns();
    prm.F = plan->F; prm.T = plan->T; prm.W = plan->W; prm.ref = plan->ref; prm.part = plan->part;
    prm.n_blocks = (int)((N + kTilesPerUnit * kTileRows - 1) / (kTilesPerUnit * kTileRows));
    prm.gathers = plan->d_gathers;
    prm.n_gathers = plan->h.n_gathers;
    if (tiled) prm.total_work = (long long)B * H * prm.n_blocks;
    const int nsm = sm_count(dev);
    if (nsm <= 0) { set_error("vdit_attn_fwd: cannot query SM count"); return VDIT_ERR_CUDA; }
    const long long grid = prm.total_work < nsm ? prm.total_work : nsm;
    const long long gwork = gathered ? (long long)B * H * plan->h.n_gathers : 0;
    if (grid <= 0 && gwork <= 0) return VDIT_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_fails_by_hook()) {
        set_error("vdit_attn_fwd: launch failure injected by vdit_set_launch_fail_after");
        return VDIT_ERR_CUDA;
    }
    if (grid > 0) {
        if (D == 128 && !tiled) {
            VDIT_CUDA_TRY((prepare_kernel<128, kModeAligned>(dev)));
            attn_fwd_kernel<128, kModeAligned><<<(unsigned)grid, kThreads, kSmemRequest, s>>>(tq, tk, tv, prm);
        } else if (D == 64 && !tiled) {
            VDIT_CUDA_TRY((prepare_kernel<64, kModeAligned>(dev)));
            attn_fwd_kernel<64, kModeAligned><<<(unsigned)grid, kThreads, kSmemRequest, s>>>(tq, tk, tv, prm);
        } else if (D == 128) {
            VDIT_CUDA_TRY((prepare_kernel<128, kModeTiled>(dev)));
            attn_fwd_kernel<128, kModeTiled><<<(unsigned)grid, kThreads, kSmemRequest, s>>>(tq, tk, tv, prm);
        } else {
            VDIT_CUDA_TRY((prepare_kernel<64, kModeTiled>(dev)));
            attn_fwd_kernel<64, kModeTiled><<<(unsigned)grid, kThreads, kSmemRequest, s>>>(tq, tk, tv, prm);
        }
        VDIT_CUDA_TRY(cudaGetLastError());
    }
    if (gwork > 0) {
        // the gathered tiles: a programmatic dependent of the launch above (which
        // lets it place CTAs once every CTA of that launch runs), so its CTAs take
        // the SMs that launch leaves at its end
        Params pg = prm;
        pg.total_work = gwork;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(gwork < nsm ? gwork : nsm));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemRequest;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = grid > 0 ? 1 : 0;
        if (D == 128) {
            VDIT_CUDA_TRY((prepare_kernel<128, kModeGathered>(dev)));
            VDIT_CUDA_TRY(cudaLaunchKernelEx(&cfg, attn_fwd_kernel<128, kModeGathered>, tq16, tk, tv, pg));
        } else {
            VDIT_CUDA_TRY((prepare_kernel<64, kModeGathered>(dev)));
            VDIT_CUDA_TRY(cudaLaunchKernelEx(&cfg, attn_fwd_kernel<64, kModeGathered>, tq16, tk, tv, pg));
        }
    }
    return VDIT_OK;
}

size_t two_pass_bytes(int32_t B, int32_t H, long long N, int32_t D) {
    const size_t rows = (size_t)B * H * (size_t)N;
    auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    return 2 * (al(rows * D * 4) + al(rows * 4));
}

}  // namespace

extern "C" vdit_status vdit_attn_fwd(const vdit_plan *plan, const void *q, const void *k,
                                     const void *v, void *o, int32_t o_dtype, float *lse,
                                     int32_t B, int32_t H, int32_t D, const int64_t q_strides[3],
                                     const int64_t k_strides[3], const int64_t v_strides[3],
                                     const int64_t o_strides[3], float scale, const float *k_mean,
                                     const float *k_rmax, const uint8_t *eligible, int32_t mode,
                                     void *stream) {
    return attn_fwd_impl(plan, q, k, v, o, o_dtype, lse, B, H, D, q_strides, k_strides, v_strides,
                         o_strides, scale, k_mean, k_rmax, eligible, nullptr, nullptr, mode, stream);
}

extern "C" vdit_status vdit_attn_fwd_framed(const vdit_plan *plan, const void *q, const void *k,
                                            const void *v, void *o, int32_t o_dtype, float *lse,
                                            int32_t B, int32_t H, int32_t D,
                                            const int64_t q_strides[3], const int64_t k_strides[3],
                                            const int64_t v_strides[3], const int64_t o_strides[3],
                                            float scale, const float *k_mean, const float *seg_rmax,
                                            const uint8_t *seg_eligible, int32_t mode,
                                            void *stream) {
    if (mode != VDIT_MODE_FORCE_ONLINE && (!k_mean || !seg_rmax)) {
        clear_error();
        set_error("vdit_attn_fwd_framed: k_mean and seg_rmax are required unless mode is FORCE_ONLINE");
        return VDIT_ERR_INVALID;
    }
    if (mode == VDIT_MODE_AUTO && !seg_eligible) {
        clear_error();
        set_error("vdit_attn_fwd_framed: seg_eligible is required in AUTO mode");
        return VDIT_ERR_INVALID;
    }
    // the per-head arguments are replaced by the per-segment ones; pass non-null
    // placeholders through the shared validation, the kernel reads the segment arrays
    return attn_fwd_impl(plan, q, k, v, o, o_dtype, lse, B, H, D, q_strides, k_strides, v_strides,
                         o_strides, scale, k_mean, seg_rmax, seg_eligible, seg_rmax, seg_eligible,
                         mode, stream);
}

extern "C" vdit_status vdit_attn_fwd_tiles128(const vdit_plan *plan, const void *q, const void *k,
                                              const void *v, void *o, int32_t o_dtype, float *lse,
                                              int32_t B, int32_t H, int32_t D, const int64_t q_strides[3],
                                              const int64_t k_strides[3], const int64_t v_strides[3],
                                              const int64_t o_strides[3], float scale, const float *k_mean,
                                              const float *k_rmax, const uint8_t *eligible, int32_t mode,
                                              void *stream) {
    return attn_fwd_impl(plan, q, k, v, o, o_dtype, lse, B, H, D, q_strides, k_strides, v_strides,
                         o_strides, scale, k_mean, k_rmax, eligible, nullptr, nullptr, mode, stream, true);
}

extern "C" size_t vdit_attn_two_pass_workspace_size(int32_t B, int32_t H, int32_t N, int32_t D) {
    if (B < 1 || H < 1 || N < 1 || D < 1) return 0;
    return two_pass_bytes(B, H, N, D);
}

extern "C" vdit_status vdit_attn_fwd_two_pass(const vdit_plan *plan_window, const vdit_plan *plan_reference,
                                              const void *q, const void *k, const void *v, void *o,
                                              int32_t o_dtype, float *lse, int32_t B, int32_t H, int32_t D,
                                              const int64_t q_strides[3], const int64_t k_strides[3],
                                              const int64_t v_strides[3], const int64_t o_strides[3],
                                              float scale, const float *k_mean, const float *k_rmax,
                                              const uint8_t *eligible, int32_t mode, int32_t tiles,
                                              void *workspace, size_t workspace_bytes, void *stream) {
    clear_error();
    if (!plan_window || !plan_reference) {
        set_error("vdit_attn_fwd_two_pass: plan is NULL");
        return VDIT_ERR_INVALID;
    }
    const vdit_plan *a = plan_window, *b = plan_reference;
    if (a->part != VDIT_PART_WINDOW || b->part != VDIT_PART_REFERENCE || a->F != b->F || a->T != b->T ||
        a->W != b->W || a->ref != b->ref || a->device != b->device) {
        set_error("vdit_attn_fwd_two_pass: needs the window part and the reference part of one mask");
        return VDIT_ERR_INVALID;
    }
    if (tiles != VDIT_TILES_FRAME && tiles != VDIT_TILES_128) {
        set_error("vdit_attn_fwd_two_pass: tiles=%d invalid", tiles);
        return VDIT_ERR_INVALID;
    }
    if (!o || !o_strides || (o_dtype != VDIT_O_BF16 && o_dtype != VDIT_O_F32) || B < 1 || H < 1 ||
        (D != 64 && D != 128)) {
        set_error("vdit_attn_fwd_two_pass: invalid output, sizes or o_dtype");
        return D == 64 || D == 128 ? VDIT_ERR_INVALID : VDIT_ERR_UNSUPPORTED;
    }
    const int oal = o_dtype == VDIT_O_F32 ? 4 : 8;
    for (int i = 0; i < 3; ++i)
        if (o_strides[i] <= 0 || o_strides[i] % oal != 0) {
            set_error("vdit_attn_fwd_two_pass: o strides must be positive multiples of 16 bytes");
            return VDIT_ERR_INVALID;
        }
    if (!aligned16(o)) { set_error("vdit_attn_fwd_two_pass: o must be 16-byte aligned"); return VDIT_ERR_INVALID; }
    const long long N = a->N;
    const size_t need = two_pass_bytes(B, H, N, D);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) {
        set_error("vdit_attn_fwd_two_pass: workspace needs %zu bytes, 256-byte aligned (got %zu)", need,
                  workspace_bytes);
        return VDIT_ERR_INVALID;
    }
    const size_t rows = (size_t)B * H * (size_t)N;
    auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    uint8_t *w = static_cast<uint8_t *>(workspace);
    float *oa = reinterpret_cast<float *>(w);
    float *la = reinterpret_cast<float *>(w + al(rows * D * 4));
    float *ob = reinterpret_cast<float *>(w + al(rows * D * 4) + al(rows * 4));
    float *lb = reinterpret_cast<float *>(w + 2 * al(rows * D * 4) + al(rows * 4));
    const int64_t dst[3] = {(int64_t)H * N * D, (int64_t)N * D, (int64_t)D};
    const bool tiled = tiles == VDIT_TILES_128;
    vdit_status st = attn_fwd_impl(a, q, k, v, oa, VDIT_O_F32, la, B, H, D, q_strides, k_strides, v_strides,
                                   dst, scale, k_mean, k_rmax, eligible, nullptr, nullptr, mode, stream, tiled);
    if (st != VDIT_OK) return st;
    st = attn_fwd_impl(b, q, k, v, ob, VDIT_O_F32, lb, B, H, D, q_strides, k_strides, v_strides, dst, scale,
                       k_mean, k_rmax, eligible, nullptr, nullptr, mode, stream, tiled);
    if (st != VDIT_OK) return st;
    const int nsm = sm_count(a->device);
    const long long blocks = ((long long)rows + 7) / 8;   // 8 warps (rows) per block
    const long long grid = blocks < 16LL * nsm ? blocks : 16LL * nsm;
    merge_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        oa, la, ob, lb, b->d_frame_runs, b->T, (int)N, H, (long long)rows, D, o, o_strides[0], o_strides[1],
        o_strides[2], o_dtype == VDIT_O_F32, lse);
    VDIT_CUDA_TRY(cudaGetLastError());
    return VDIT_OK;
}

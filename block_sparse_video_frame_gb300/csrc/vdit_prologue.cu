// Fused pre-attention chain for sm_103a: RMSNorm, q/k/v projection, rotary
// embedding and head packing, written straight into attention's [B, H, N, D]
// layout.
//
// "HeyGen x Google Cloud: Bringing Avatar IV to TPUs", "Layout Is the ABI"
// (Fig. 5): the chain that produces attention's inputs is fused into one
// kernel whose output buffer is the next consumer's input buffer, so no repack
// copies remain between the projections and that consumer.
//
// GB300 design. RMSNorm's per-row scale commutes with the contraction,
//   z = W (gamma . x / rms(x)) = (1 / rms(x)) * (W diag(gamma)) x,
// so the gain folds into the weights once (fold_gamma_kernel) and each call
// runs:
//   rms_kernel   one warp per token row: 1/rms in fp32 (HBM-bound pre-pass)
//   qkv_gemm     persistent tcgen05 GEMM, x [rows, C] . W'^T [C, 3HD], on CTA
//                pairs (clusters of 2, one CTA per SM): a pair computes a
//                256 x 256 output tile with cta_group::2 MMAs (M = 256 over
//                both SMs, N = 256), each CTA staging its own 128 x rows and
//                half of the 256 W' rows, so per SM only 32 KB cross from L2
//                per 64-deep K stage (48 KB for a lone 128 x 256 tile)
//     warp 0     TMEM allocator (both CTAs); on rank 0 the single-thread MMA
//                issuer. Two 256-column fp32 accumulators per CTA (512 TMEM
//                columns) so one tile's epilogue overlaps the next tile's MMAs
//     warp 1     TMA producer: 6-stage ring of x (128 x 64) and W' (128 x 64)
//                tiles, bf16, 128-byte swizzle; both CTAs' loads complete on
//                rank 0's stage barrier, where the MMA issuer waits
//     warps 2-5  epilogue: thread = output row (TMEM lane of its CTA); 1/rms
//                scale, rotation of q and k heads by the angle table, bf16
//                rounding, 128-byte-swizzled staging in shared memory, TMA
//                stores into q, k, v ([B, H, N, D]); rows past N are clipped
// Every wait is bounded in time; on expiry the CTA records a site code in the
// workspace status word, both CTAs drain their in-flight copies and MMAs, free
// TMEM and exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "vdit_internal.h"
#include "vdit_ptx.cuh"

namespace vdit {
namespace {

using namespace ptx;

// ---------------------------------------------------------------- extra PTX
// Loads whose completion is signalled on an mbarrier of either CTA of the pair
// (cluster address), for the CTA-pair MMA.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// 4-D tiled TMA store of one box from shared memory (bulk-group completion).
// Coordinates are non-negative; the parts of the box outside the tensor are
// not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Named barrier over the epilogue's 128 threads.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Named barrier over the epilogue's 128 threads that also returns, to every
// one of them, whether any thread passed a non-zero `bad`.
__device__ __forceinline__ bool epi_sync_any(uint32_t bad) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(bad)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// ---------------------------------------------------------------- CTA pair (cluster of 2)
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Arrive on an mbarrier of another CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// 32-bit store to another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Count `bytes` as arrived on a local mbarrier's current phase without a copy.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// tcgen05 over the CTA pair: allocation (one warp in each CTA), MMA issued by
// one thread of the even CTA, commits that arrive at the same barrier offset
// in both CTAs.
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma2_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma2_commit_both(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// Bounded waits. The GEMM's waits are short (one K stage, one tile), so the
// slow path reads the clock after every failed poll (each try_wait already
// suspends the thread for a while): a wait that outlasts the bound always
// expires, whatever the bound. On expiry, or when another thread of the CTA has
// given up (*abort), it records `site` in the status word (first writer wins),
// raises *abort and returns false.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort, int *status,
                                       int site, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > limit_ns) {
            *abort = 1;
            atomicCAS(status, 0, site);
            return false;
        }
    }
}
// One thread.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile int *abort, int *status,
                                      int site, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort, status, site, limit_ns);
}
// Whole warp, warp-uniform result.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int *status, int site, uint64_t limit_ns) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const bool r = wait_slow(bar, parity, abort, status, site, limit_ns);
    return __all_sync(0xffffffffu, r);
}

// ---------------------------------------------------------------- geometry
// A CTA pair computes a 256 x 256 output tile: CTA rank r holds x rows
// [m0 + 128 r, m0 + 128 r + 128) and W' rows (output columns) [n0 + 128 r, +128)
// of every K stage; one thread of rank 0 issues 256 x 256 x 16 MMAs over both
// CTAs' shared memory, and each CTA's TMEM receives its own 128 rows x 256 columns.
constexpr int kRmsThreads = 512;     // 1/rms pre-pass: 16 rows in flight per block
constexpr int kBM = 128;             // output rows per CTA (TMEM lanes)
constexpr int kPairM = 256;          // output rows per CTA pair (tcgen05 M, cta_group::2)
constexpr int kBN = 256;             // output columns per tile (tcgen05 N)
constexpr int kHalfN = kBN / 2;      // W' rows staged per CTA
constexpr int kBK = 64;              // K per stage: one 128-byte swizzle atom of bf16
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kWarpMma = 0, kWarpTma = 1, kWarpEpi0 = 2;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kHalfN * kBK * 2;       // 16 KB
constexpr int kStageTx = kABytes + kBBytes;     // bytes one CTA loads per stage
constexpr int kBoxBytes = kBM * 64 * 2;         // one 128-row x 64-column bf16 store box
constexpr int kSmA = 0;
constexpr int kSmB = kSmA + kStages * kABytes;
constexpr int kSmStage = kSmB + kStages * kBBytes;   // two store boxes (one 128-column group)
constexpr int kSmBar = kSmStage + 2 * kBoxBytes;
enum : int { kBarFull = 0, kBarEmpty = kStages, kBarAccFull = 2 * kStages, kBarAccEmpty = kBarAccFull + 2,
             kBarFinal = kBarAccEmpty + 2, kNumBars = kBarFinal + 1 };
constexpr int kSmBytes = kSmBar + 8 * kNumBars + 16;
constexpr int kSmAlloc = kSmBytes + 1024;      // slack to align the base to 1024 bytes
static_assert(kSmAlloc <= 232448, "prologue GEMM shared memory exceeds the per-CTA limit");

// status-word site codes (which wait expired); distinct from the attention kernel's
enum : int { kSiteEmpty = 101, kSiteFull, kSiteAccEmpty, kSiteAccFull };

struct GemmParams {
    int B, N, H, D, C, O;        // O = 3 H D output columns
    int pairs_m, tiles_n, kb;    // 256-row blocks per batch, column tiles, K stages per tile
    int col_bands;               // column bands the tiles are walked in (see tile_of)
    long long total;             // B * pairs_m * tiles_n pair tiles
    const float *inv_rms;        // [B * N]
    const float2 *rope;          // [D/2][N] (cos, sin)
    int *status;
    unsigned long long timeout_ns;
};

// ---------------------------------------------------------------- small kernels
// w_folded[o, c] = bf16(fp32(w[o, c]) * gamma[c]) (in place allowed).
__global__ void fold_gamma_kernel(const __nv_bfloat16 *w, const float *gamma, __nv_bfloat16 *wf,
                                  long long total, int C) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const float g = gamma[i % C];
        wf[i] = __float2bfloat16_rn(__bfloat162float(w[i]) * g);
    }
}

// table[i][n] = (cos a, sin a), a = n * base^(-2i/D), evaluated in fp64.
__global__ void rope_table_kernel(float2 *table, int N, int D, double base) {
    const long long total = (long long)(D / 2) * N;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(idx / N), n = (int)(idx % N);
        const double t = pow(base, -2.0 * i / (double)D);
        double s, c;
        sincos((double)n * t, &s, &c);
        table[idx] = make_float2((float)c, (float)s);
    }
}

// inv_rms[b*N + n] = 1 / sqrt(mean_c x[b, n, c]^2 + eps), one warp per row
// (grid-stride over rows), 16-byte loads (C a multiple of 8), fp32
// accumulation in a fixed order.
__global__ void __launch_bounds__(kRmsThreads)
rms_kernel(const __nv_bfloat16 *x, long long xs0, long long xs1, int B, int N, int C, float eps,
           float *inv_rms) {
    // The GEMM that consumes inv_rms may start now: only its epilogue waits
    // for this grid (griddepcontrol.wait), its loads and MMAs overlap this pass.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x % 32;
    const long long rows = (long long)B * N;
    const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
    for (long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; row < rows;
         row += nwarps) {   // warp-uniform
        const long long b = row / N, n = row % N;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + b * xs0 + n * xs1);
        float acc = 0.f;
        auto add_sq = [&](const uint4 &u) {
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
                acc = fmaf(lo, lo, acc);
                acc = fmaf(hi, hi, acc);
            }
        };
        // batches of 8 independent 16-byte loads per lane (64 KB in flight per
        // SM at 16 warps), then the remainder one load at a time
        const int nv = C / 8;
        int v0 = 0;
        for (; v0 + 32 * 8 <= nv; v0 += 32 * 8) {
            uint4 u[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) u[j] = __ldg(src + v0 + 32 * j + lane);
#pragma unroll
            for (int j = 0; j < 8; ++j) add_sq(u[j]);
        }
        for (int v = v0 + lane; v < nv; v += 32) add_sq(__ldg(src + v));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) inv_rms[row] = 1.0f / sqrtf(acc / (float)C + eps);
    }
}

// Poll a barrier phase for at most `limit_ns` (teardown: copies and MMAs in
// flight must land before shared memory and TMEM are released).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) return false;
    }
    return true;
}

struct TileId {
    int b, mp, nt;
};
// Tile order. The output columns are walked in p.col_bands bands. Inside a band the
// column tiles go fastest, so concurrent pairs share x rows, and every 256-row block
// is visited before the next band starts. So only one band of W' has to stay in L2
// while x and the outputs stream through it, at the price of reading x once per band.
__device__ __forceinline__ TileId tile_of(const GemmParams &p, long long t) {
    const long long per_b = (long long)p.pairs_m * p.tiles_n;
    TileId id;
    id.b = (int)(t / per_b);
    const int rem = (int)(t - (long long)id.b * per_b);
    const int nb = (p.tiles_n + p.col_bands - 1) / p.col_bands;   // tiles per full band
    const int band = rem / (p.pairs_m * nb);
    const int r2 = rem - band * p.pairs_m * nb;
    const int wb = min(nb, p.tiles_n - band * nb);                // this band's width
    id.mp = r2 / wb;
    id.nt = band * nb + r2 % wb;
    return id;
}

// ---------------------------------------------------------------- the GEMM
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
qkv_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + kSmBar;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kSmBar + 8 * kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kSmBar + 8 * kNumBars + 4);
    volatile uint32_t *peer_kc = reinterpret_cast<volatile uint32_t *>(smem + kSmBar + 8 * kNumBars + 8);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();
    const bool lead = rank == 0;
    const uint64_t tlim = p.timeout_ns;
    const long long npairs = gridDim.x / 2, pair = blockIdx.x / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // rank 0's barrier counts both CTAs' bytes; rank 1's is unused
            mbar_init(bar(kBarFull + s), 1);
            mbar_init(bar(kBarEmpty + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(kBarAccFull + a), 1);
            mbar_init(bar(kBarAccEmpty + a), 8);   // the epilogue warps of both CTAs
        }
        mbar_init(bar(kBarFinal), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc2(smem_addr(tmem_slot), 512);
        tmem_relinquish2();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised before any cross-CTA arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    uint32_t issued = 0;   // K stages this CTA's producer loaded

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            uint32_t kc = 0;  // stages issued
            bool ok = true;
            for (long long t = pair; ok && t < p.total; t += npairs) {
                const TileId id = tile_of(p, t);
                const int row = id.mp * kPairM + (int)rank * kBM;
                const int col = id.nt * kBN + (int)rank * kHalfN;
                for (int kb = 0; kb < p.kb; ++kb, ++kc) {
                    const int s = kc % kStages;
                    if (!(ok = wait1(bar(kBarEmpty + s), ((kc / kStages) & 1) ^ 1, abort_flag,
                                     p.status, kSiteEmpty, tlim)))
                        break;
                    // both CTAs' bytes complete on rank 0's barrier
                    if (lead) mbar_arrive_expect_tx(bar(kBarFull + s), 2 * kStageTx);
                    const uint32_t fb = map_to_rank(bar(kBarFull + s), 0);
                    tma_load_3d_pair(sbase + kSmA + s * kABytes, &tm_x, fb, kb * kBK, row, id.b);
                    tma_load_2d_pair(sbase + kSmB + s * kBBytes, &tm_w, fb, kb * kBK, col);
                }
            }
            issued = kc;
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer (rank 0)
        if (lead) {
            const bool leader = elect_one();
            const uint64_t dA = sdesc_sw128(sbase + kSmA, 16, 1024);
            const uint64_t dB = sdesc_sw128(sbase + kSmB, 16, 1024);
            constexpr uint32_t kIdesc = idesc_bf16(kPairM, kBN, false);
            uint32_t kc = 0, tc = 0;
            bool ok = true;
            for (long long t = pair; ok && t < p.total; t += npairs, ++tc) {
                const uint32_t buf = tc & 1, use = tc >> 1;
                if (!(ok = wait_warp(bar(kBarAccEmpty + buf), (use & 1) ^ 1, abort_flag, p.status,
                                     kSiteAccEmpty, tlim)))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + buf * kBN;
                for (int kb = 0; kb < p.kb; ++kb, ++kc) {
                    const int s = kc % kStages;
                    if (!(ok = wait_warp(bar(kBarFull + s), (kc / kStages) & 1, abort_flag, p.status,
                                         kSiteFull, tlim)))
                        break;
                    tc_fence_after();
                    if (leader) {
                        const uint64_t a0 = dA + (uint64_t)(s * (kABytes >> 4));
                        const uint64_t b0 = dB + (uint64_t)(s * (kBBytes >> 4));
#pragma unroll
                        for (int ks = 0; ks < kBK / 16; ++ks)
                            mma2_ss(d, a0 + ks * 2, b0 + ks * 2, kIdesc, (kb | ks) != 0 ? 1u : 0u);
                        mma2_commit_both(bar(kBarEmpty + s));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (leader) mma2_commit_both(bar(kBarAccFull + buf));
                __syncwarp();
            }
            // drain: all issued MMAs complete (in both CTAs' TMEM) before the
            // closing cluster barrier, after which both CTAs release TMEM
            if (leader) mma2_commit_both(bar(kBarFinal));
            __syncwarp();
            drain_wait(bar(kBarFinal), 0, kDefaultWaitLimitNs);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int qd = warp % 4;                     // TMEM lane quadrant of this warp
        const int r = qd * 32 + lane;                // row within the tile
        const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
        const bool store_thread = warp == kWarpEpi0 && lane == 0;
        const int HD = p.H * p.D, half = p.D / 2;
        const uint32_t row_smem = sbase + kSmStage + (uint32_t)r * 128;
        const uint32_t swz = (uint32_t)(r & 7);
        uint32_t tc = 0;
        // rank 1 hands its accumulator back on rank 0's barrier
        const uint32_t acc_empty0 = lead ? bar(kBarAccEmpty) : map_to_rank(bar(kBarAccEmpty), 0);
        for (long long t = pair; t < p.total; t += npairs, ++tc) {
            const TileId id = tile_of(p, t);
            const uint32_t buf = tc & 1, use = tc >> 1;
            const bool got = wait_warp(bar(kBarAccFull + buf), use & 1, abort_flag, p.status,
                                            kSiteAccFull, tlim);
            if (epi_sync_any(got ? 0u : 1u)) break;  // uniform over the four warps
            tc_fence_after();
            const int row0 = id.mp * kPairM + (int)rank * kBM;   // first row of this CTA's half
            const int n = row0 + r;
            const bool live = n < p.N;
            if (tc == 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // 1/rms pre-pass done
            const float sc = live ? p.inv_rms[(long long)id.b * p.N + n] : 0.f;
            const uint32_t tacc = tmem + buf * kBN + lane_off;
            const int col_t = id.nt * kBN;
            const int ngroups = min(kBN / 128, (p.O - col_t + 127) / 128);
            for (int g = 0; g < ngroups; ++g) {
                const int col0 = col_t + g * 128;        // first output column of the group
                if (store_thread) bulk_wait_read0();   // staging free: previous stores have read it
                epi_sync();
#pragma unroll 1
                for (int s2 = 0; s2 < 2; ++s2) {
                    // D = 128: one head per group, pairs (32 s2 + j, 64 + 32 s2 + j).
                    // D = 64: head s2 of the group, pairs (j, 32 + j).
                    const int head_col = p.D == 128 ? 0 : 64 * s2;
                    const int lo_col = p.D == 128 ? 32 * s2 : 64 * s2;
                    const int o = col0 + head_col;
                    if (o >= p.O) continue;               // warp-uniform
                    const int part = o / HD;
                    uint32_t lo[32], hi[32], plo[16], phi[16];
                    tmem_ld32(tacc + g * 128 + lo_col, lo);
                    tmem_ld32(tacc + g * 128 + lo_col + half, hi);
                    if (part < 2) {
                        const int i0 = lo_col - head_col;   // rotation pair of column j = 0
                        const float2 *cs = p.rope + (size_t)i0 * p.N + (live ? n : 0);
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float2 t0 = cs[(size_t)j * p.N], t1 = cs[(size_t)(j + 1) * p.N];
                            const float a0 = __uint_as_float(lo[j]) * sc, b0 = __uint_as_float(hi[j]) * sc;
                            const float a1 = __uint_as_float(lo[j + 1]) * sc,
                                        b1 = __uint_as_float(hi[j + 1]) * sc;
                            plo[j / 2] = pack_bf16(fmaf(a0, t0.x, -b0 * t0.y), fmaf(a1, t1.x, -b1 * t1.y));
                            phi[j / 2] = pack_bf16(fmaf(a0, t0.y, b0 * t0.x), fmaf(a1, t1.y, b1 * t1.x));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            plo[j / 2] = pack_bf16(__uint_as_float(lo[j]) * sc, __uint_as_float(lo[j + 1]) * sc);
                            phi[j / 2] = pack_bf16(__uint_as_float(hi[j]) * sc, __uint_as_float(hi[j + 1]) * sc);
                        }
                    }
                    // staging: D = 128 puts the low half in box 0 and the high half in
                    // box 1 (chunks 4 s2 ..); D = 64 puts head s2 in box s2 (chunks 0-3, 4-7)
                    const uint32_t lo_box = p.D == 128 ? 0u : (uint32_t)s2;
                    const uint32_t hi_box = p.D == 128 ? 1u : (uint32_t)s2;
                    const uint32_t lo_ch = p.D == 128 ? 4u * s2 : 0u, hi_ch = p.D == 128 ? 4u * s2 : 4u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        st_shared_v4(row_smem + lo_box * kBoxBytes + (((lo_ch + c) ^ swz) << 4),
                                     plo[4 * c], plo[4 * c + 1], plo[4 * c + 2], plo[4 * c + 3]);
                        st_shared_v4(row_smem + hi_box * kBoxBytes + (((hi_ch + c) ^ swz) << 4),
                                     phi[4 * c], phi[4 * c + 1], phi[4 * c + 2], phi[4 * c + 3]);
                    }
                }
                if (g == ngroups - 1) {
                    // every TMEM read of this accumulator is done: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (lead) mbar_arrive(bar(kBarAccEmpty + buf));
                        else mbar_arrive_remote(acc_empty0 + 8u * buf);
                    }
                }
                fence_async_smem();
                epi_sync();
                if (store_thread && row0 < p.N) {
#pragma unroll 1
                    for (int bx = 0; bx < 2; ++bx) {
                        const int o = col0 + 64 * bx;       // first output column of the box
                        if (o >= p.O) continue;
                        const int part = o / HD, h = (o % HD) / p.D, d0 = o % p.D;
                        const CUtensorMap *m = part == 0 ? &tm_q : (part == 1 ? &tm_k : &tm_v);
                        tma_store_4d(m, sbase + kSmStage + bx * kBoxBytes, d0, row0, h, id.b);
                    }
                    bulk_commit();
                }
            }
        }
        if (store_thread) bulk_wait0();
    }

    // Teardown. Every load of both CTAs completes on rank 0's stage barriers, so
    // rank 0 drains them for both: rank 1 reports how many stages it loaded,
    // and where an early exit left the two counts one phase apart rank 0
    // supplies the missing expectation (rank 1's bytes arrive unexpected) or
    // the missing bytes (rank 1 never loaded), then waits for the last phase.
    if (!lead && warp == kWarpTma && lane == 0)
        st_cluster_u32(map_to_rank(smem_addr(const_cast<uint32_t *>(peer_kc)), 0), issued);
    tc_fence_before();
    cluster_sync();   // all roles done; MMAs drained; rank 1's count visible
    if (lead && warp == kWarpTma && lane == 0) {
        const uint32_t kc1 = *peer_kc;
        for (int s = 0; s < kStages; ++s) {
            const uint32_t n0 = issued / kStages + ((uint32_t)s < issued % kStages ? 1u : 0u);
            const uint32_t n1 = kc1 / kStages + ((uint32_t)s < kc1 % kStages ? 1u : 0u);
            if (n1 > n0) mbar_arrive_expect_tx(bar(kBarFull + s), kStageTx);
            else if (n0 > n1) mbar_complete_tx(bar(kBarFull + s), kStageTx);
            const uint32_t n = n0 > n1 ? n0 : n1;
            if (n > 0) drain_wait(bar(kBarFull + s), (n - 1) & 1, kDefaultWaitLimitNs);
        }
    }
    cluster_sync();   // no copy, arrival or MMA of either CTA is outstanding
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc2(tmem, 512);
    }
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

// bf16 tensor map, 128-byte swizzle; dims/strides innermost first (strides in bytes).
bool encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

cudaError_t prepare_gemm(int device) {
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> g(mu);
    if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(qkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
    if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
    return e;
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

// Co-resident CTA pairs of the GEMM on this device (one pair per two SMs
// where the GPCs allow it): the persistent grid size.
int max_pairs(int device) {
    static std::mutex mu;
    static int cache[64] = {};
    std::lock_guard<std::mutex> g(mu);
    if (device < 0 || device >= 64) return 0;
    if (cache[device] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmAlloc;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, qkv_gemm_kernel, &cfg) == cudaSuccess) cache[device] = n;
    }
    return cache[device];
}

constexpr size_t kWsHeader = 256;   // status word, padded

unsigned grid_for(long long work, int per_block) {
    long long g = (work + per_block - 1) / per_block;
    if (g > 65536) g = 65536;
    return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace vdit

using namespace vdit;

extern "C" vdit_status vdit_qkv_fold_gamma(const void *w, const float *gamma, void *w_folded,
                                           int64_t rows, int32_t C, void *stream) {
    clear_error();
    if (!w || !gamma || !w_folded) {
        set_error("vdit_qkv_fold_gamma: NULL pointer argument");
        return VDIT_ERR_INVALID;
    }
    if (rows < 1 || C < 1) {
        set_error("vdit_qkv_fold_gamma: rows=%lld C=%d must be >= 1", (long long)rows, C);
        return VDIT_ERR_INVALID;
    }
    const long long total = (long long)rows * C;
    fold_gamma_kernel<<<grid_for(total, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(w), gamma, static_cast<__nv_bfloat16 *>(w_folded), total, C);
    VDIT_CUDA_TRY(cudaGetLastError());
    return VDIT_OK;
}

extern "C" vdit_status vdit_rope_table(float *table, int32_t N, int32_t D, double base, void *stream) {
    clear_error();
    if (!table) { set_error("vdit_rope_table: table is NULL"); return VDIT_ERR_INVALID; }
    if (N < 1 || D < 2 || D % 2 != 0) {
        set_error("vdit_rope_table: N=%d must be >= 1 and D=%d even and >= 2", N, D);
        return VDIT_ERR_INVALID;
    }
    if (!(base > 0.0 && base <= 1.7976931348623157e308)) { set_error("vdit_rope_table: base must be finite and > 0"); return VDIT_ERR_INVALID; }
    if (reinterpret_cast<uintptr_t>(table) & 7u) {
        set_error("vdit_rope_table: table must be 8-byte aligned");
        return VDIT_ERR_INVALID;
    }
    const long long total = (long long)(D / 2) * N;
    rope_table_kernel<<<grid_for(total, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<float2 *>(table), N, D, base);
    VDIT_CUDA_TRY(cudaGetLastError());
    return VDIT_OK;
}

extern "C" size_t vdit_qkv_workspace_size(int32_t B, int32_t N) {
    if (B < 1 || N < 1) return 0;
    return kWsHeader + (((size_t)B * (size_t)N * sizeof(float) + 255) & ~(size_t)255);
}

extern "C" vdit_status vdit_qkv_prologue(const void *x, const int64_t x_strides[2],
                                         const void *w_folded, const float *rope, void *q, void *k,
                                         void *v, const int64_t q_strides[3],
                                         const int64_t k_strides[3], const int64_t v_strides[3],
                                         int32_t B, int32_t N, int32_t C, int32_t H, int32_t D,
                                         float eps, void *workspace, size_t workspace_bytes,
                                         void *stream) {
    clear_error();
    if (!x || !x_strides || !w_folded || !rope || !q || !k || !v || !q_strides || !k_strides ||
        !v_strides || !workspace) {
        set_error("vdit_qkv_prologue: NULL pointer argument");
        return VDIT_ERR_INVALID;
    }
    if (B < 1 || N < 1 || H < 1 || C < 8) {
        set_error("vdit_qkv_prologue: B=%d N=%d H=%d must be >= 1 and C=%d >= 8", B, N, H, C);
        return VDIT_ERR_INVALID;
    }
    if (D != 64 && D != 128) {
        set_error("vdit_qkv_prologue: head dim D=%d not supported (64 or 128)", D);
        return VDIT_ERR_UNSUPPORTED;
    }
    if (C % 8 != 0) { set_error("vdit_qkv_prologue: C=%d must be a multiple of 8", C); return VDIT_ERR_INVALID; }
    const long long O = 3ll * H * D;
    if (O > (1ll << 30)) { set_error("vdit_qkv_prologue: 3*H*D too large"); return VDIT_ERR_INVALID; }
    if (!(eps >= 0.f && eps <= 3.402823466e38f)) { set_error("vdit_qkv_prologue: eps must be finite and >= 0"); return VDIT_ERR_INVALID; }
    for (int i = 0; i < 2; ++i)
        if (x_strides[i] <= 0 || x_strides[i] % 8 != 0 || x_strides[i] >= (1ll << 38)) {
            set_error("vdit_qkv_prologue: x strides must be positive multiples of 8 elements");
            return VDIT_ERR_INVALID;
        }
    if (x_strides[1] < C) { set_error("vdit_qkv_prologue: x row stride is below C"); return VDIT_ERR_INVALID; }
    const int64_t *sts[3] = {q_strides, k_strides, v_strides};
    for (int t = 0; t < 3; ++t)
        for (int i = 0; i < 3; ++i)
            if (sts[t][i] <= 0 || sts[t][i] % 8 != 0 || sts[t][i] >= (1ll << 38)) {
                set_error("vdit_qkv_prologue: q/k/v strides must be positive multiples of 8 elements");
                return VDIT_ERR_INVALID;
            }
    if (!aligned16(x) || !aligned16(w_folded) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(rope) || !aligned16(workspace)) {
        set_error("vdit_qkv_prologue: x, w_folded, rope, q, k, v and workspace must be 16-byte aligned");
        return VDIT_ERR_INVALID;
    }
    if (workspace_bytes < vdit_qkv_workspace_size(B, N)) {
        set_error("vdit_qkv_prologue: workspace of %zu bytes is below the %zu required", workspace_bytes,
                  vdit_qkv_workspace_size(B, N));
        return VDIT_ERR_INVALID;
    }
    int dev = -1;
    VDIT_CUDA_TRY(cudaGetDevice(&dev));

    CUtensorMap tx, tw, tq, tk, tv;
    {
        const cuuint64_t xd[3] = {(cuuint64_t)C, (cuuint64_t)N, (cuuint64_t)B};
        const cuuint64_t xs[2] = {(cuuint64_t)x_strides[1] * 2, (cuuint64_t)x_strides[0] * 2};
        const cuuint32_t xb[3] = {64, 128, 1};
        const cuuint64_t wd[2] = {(cuuint64_t)C, (cuuint64_t)O};
        const cuuint64_t ws[1] = {(cuuint64_t)C * 2};
        const cuuint32_t wb[2] = {64, (cuuint32_t)kHalfN};
        const cuuint32_t ob[4] = {64, 128, 1, 1};
        const cuuint64_t od[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
        bool ok = encode(&tx, x, 3, xd, xs, xb) && encode(&tw, w_folded, 2, wd, ws, wb);
        void *outs[3] = {q, k, v};
        CUtensorMap *maps[3] = {&tq, &tk, &tv};
        for (int t = 0; ok && t < 3; ++t) {
            const cuuint64_t os[3] = {(cuuint64_t)sts[t][2] * 2, (cuuint64_t)sts[t][1] * 2,
                                      (cuuint64_t)sts[t][0] * 2};
            ok = encode(maps[t], outs[t], 4, od, os, ob);
        }
        if (!ok) {
            set_error("vdit_qkv_prologue: cuTensorMapEncodeTiled failed (alignment/strides or driver entry point)");
            return VDIT_ERR_INVALID;
        }
    }
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    float *inv_rms = reinterpret_cast<float *>(wsb + kWsHeader);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const long long rows = (long long)B * N;
    // One resident block per SM (grid-stride over rows), small enough to share
    // each SM with a GEMM CTA, which launches as soon as every block has started.
    const int nsm = sm_count(dev);
    if (nsm <= 0) { set_error("vdit_qkv_prologue: cannot query SM count"); return VDIT_ERR_CUDA; }
    const long long rms_blocks = (rows + kRmsThreads / 32 - 1) / (kRmsThreads / 32);
    rms_kernel<<<(unsigned)(rms_blocks < nsm ? rms_blocks : nsm), kRmsThreads, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(x), x_strides[0], x_strides[1], B, N, C, eps, inv_rms);
    VDIT_CUDA_TRY(cudaGetLastError());

    GemmParams prm;
    prm.B = B; prm.N = N; prm.H = H; prm.D = D; prm.C = C; prm.O = (int)O;
    prm.pairs_m = (N + kPairM - 1) / kPairM;
    prm.tiles_n = (int)((O + kBN - 1) / kBN);
    prm.kb = (C + kBK - 1) / kBK;
    prm.total = (long long)B * prm.pairs_m * prm.tiles_n;
    {
        // one band per 24 MB of W' (three for the 9216 x 3072 projection): a band of W'
        // then stays in L2 beside the streaming x and outputs. DRAM reads at that
        // size: 1.83 GB in one band, 1.34 GB in two, 1.06 GB in three.
        const long long w_bytes = O * (long long)C * 2;
        const long long band_bytes = 24ll << 20;
        const long long bands = (w_bytes + band_bytes - 1) / band_bytes;
        prm.col_bands = (int)(bands < 1 ? 1 : (bands > prm.tiles_n ? prm.tiles_n : bands));
    }
    prm.inv_rms = inv_rms;
    prm.rope = reinterpret_cast<const float2 *>(rope);
    prm.status = reinterpret_cast<int *>(wsb);
    prm.timeout_ns = wait_limit_ns();
    VDIT_CUDA_TRY(prepare_gemm(dev));
    const int pairs = max_pairs(dev);
    if (pairs <= 0) { set_error("vdit_qkv_prologue: no CTA pair fits on this device"); return VDIT_ERR_CUDA; }
    const long long grid = 2 * (prm.total < pairs ? prm.total : pairs);
    // Programmatic dependent launch on the pre-pass (cluster shape from the kernel).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    VDIT_CUDA_TRY(cudaLaunchKernelEx(&cfg, qkv_gemm_kernel, tx, tw, tq, tk, tv, prm));
    return VDIT_OK;
}

extern "C" vdit_status vdit_qkv_status(void *workspace, void *stream, int32_t *code) {
    clear_error();
    if (!workspace) { set_error("vdit_qkv_status: workspace is NULL"); return VDIT_ERR_INVALID; }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    VDIT_CUDA_TRY(cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s));
    VDIT_CUDA_TRY(cudaStreamSynchronize(s));
    if (code) *code = word;
    if (word != 0) {
        VDIT_CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof word, s));
        VDIT_CUDA_TRY(cudaStreamSynchronize(s));
        set_error("vdit_qkv_prologue: a bounded wait expired (site %d)", word);
        return VDIT_ERR_TIMEOUT;
    }
    return VDIT_OK;
}

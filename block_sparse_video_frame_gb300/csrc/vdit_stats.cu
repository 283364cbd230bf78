// Per-head key statistics and static-max eligibility.
//
// "HeyGen x Google Cloud: Bringing Avatar IV to TPUs", "Unchaining the
// Softmax": a few numbers per head, computed before attention, give every query
// row an upper bound on its logits before its first key tile. Centring the keys
// on their mean tightens the bound and leaves the softmax unchanged; a head with a
// loose bound runs online softmax instead. This file computes, per (b, h):
//   c    = (1/N) sum_j k_j          R  = max_j |k_j - c|
//   Qm   = max_i |q_i|              G  = 2 * scale * Qm * R,  eligible = G <= tau
// HBM-bound: K is read twice (the second read comes from L2 only while K fits
// there; at 720p only the last heads of the first pass are still there), Q once.
// Four launches, every reduction in a fixed order (bitwise reproducible):
//   stats_pass1    per chunk of 512 rows: column sums of K, max |q|^2
//   stats_mean     c = (sum of the chunk column sums) / N, per head
//   stats_pass2    per chunk: max |k - c|^2
//   stats_finalize R, Qm, G, eligibility
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "vdit_internal.h"

namespace vdit {
namespace {

constexpr int kRowsPerChunk = 512;
constexpr int kStatsThreads = 256;
constexpr int kStatsWarps = kStatsThreads / 32;

struct StatsArgs {
    const __nv_bfloat16 *q, *k;
    long long qs0, qs1, qs2, ks0, ks1, ks2;
    int B, H, N, nchunk;
    int T, cpf;          // rows per frame (N when frames are not used) and chunks per frame
    float scale, tau;
    float *ws_colsum, *ws_qn2, *ws_rn2;
    float *k_mean, *k_rmax, *q_nmax, *gap;
    uint8_t *elig;
};

// Each lane loads 16 bytes (8 bf16) of a row; a row of D elements takes
// D/8 lanes, so one warp-wide load covers 32/(D/8) rows. Every warp keeps
// kUnroll such loads per tensor in flight.
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 load16(const __nv_bfloat16 *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}
// bf16 element e (0..7) of a 16-byte load, as fp32 (exact)
__device__ __forceinline__ float elem8(const uint4 &u, int e) {
    const uint32_t w = e < 2 ? u.x : e < 4 ? u.y : e < 6 ? u.z : u.w;
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// sum over the LPR lanes that hold one row (a contiguous, aligned group of lanes)
template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
__global__ void __launch_bounds__(kStatsThreads, 4) stats_pass1(StatsArgs a) {
    constexpr int LPR = D / 8;          // lanes per row
    constexpr int RPW = 32 / LPR;       // rows per warp-wide load
    __shared__ float s_col[kStatsWarps * RPW][D];
    __shared__ float s_q[kStatsWarps];
    const int chunk = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub = lane / LPR, col = (lane % LPR) * 8;
    const __nv_bfloat16 *kb = a.k + b * a.ks0 + h * a.ks1 + col;
    const __nv_bfloat16 *qb = a.q + b * a.qs0 + h * a.qs1 + col;
    const int fr = chunk / a.cpf;
    const int r0 = fr * a.T + (chunk % a.cpf) * kRowsPerChunk;
    const int r1 = min((fr + 1) * a.T, r0 + kRowsPerChunk);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float qm2 = 0.f;
    constexpr int kStep = kStatsWarps * RPW;        // rows covered by the block per load
    // warp-uniform loop bound: every lane runs the same iterations (the row
    // sums below shuffle across the whole warp); rows past the chunk load zeros
    for (int wbase = r0 + warp * RPW; wbase < r1; wbase += kStep * kUnroll) {
        // raw 16-byte loads stay packed until used (few registers, more
        // blocks per SM, more loads in flight)
        uint4 xk[kUnroll], xq[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int r = wbase + sub + u * kStep;
            if (r < r1) {
                xk[u] = load16(kb + (long long)r * a.ks2);
                xq[u] = load16(qb + (long long)r * a.qs2);
            } else {
                xk[u] = xq[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += elem8(xk[u], e);
            float sq = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float x = elem8(xq[u], e);
                sq = fmaf(x, x, sq);
            }
            qm2 = fmaxf(qm2, row_sum<LPR>(sq));
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s_col[warp * RPW + sub][col + e] = acc[e];
    qm2 = warp_max(qm2);
    if (lane == 0) s_q[warp] = qm2;
    __syncthreads();
    const size_t slot = (size_t)bh * a.nchunk + chunk;
    for (int d = threadIdx.x; d < D; d += kStatsThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kStatsWarps * RPW; ++w) t += s_col[w][d];
        a.ws_colsum[slot * D + d] = t;
    }
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int w = 0; w < kStatsWarps; ++w) m = fmaxf(m, s_q[w]);
        a.ws_qn2[slot] = m;
    }
}

// c = (1/N) * sum of the chunk column sums, chunks in ascending order.
__global__ void stats_mean(StatsArgs a, int D) {
    const int bh = blockIdx.x;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float t = 0.f;
        for (int c = 0; c < a.nchunk; ++c) t += a.ws_colsum[((size_t)bh * a.nchunk + c) * D + d];
        a.k_mean[(size_t)bh * D + d] = t / (float)a.N;
    }
}

// Pass 2 reads one tensor where pass 1 reads two: twice the unroll keeps as many
// 16-byte loads in flight per warp, packed until used.
constexpr int kUnroll2 = 2 * kUnroll;

template <int D>
__global__ void __launch_bounds__(kStatsThreads, 4) stats_pass2(StatsArgs a) {
    constexpr int LPR = D / 8;
    constexpr int RPW = 32 / LPR;
    __shared__ float s_r[kStatsWarps];
    // Heads in reverse order: pass 1 walked them forward, so the keys of its last
    // heads are still in L2 when this pass starts (each head's result is the same in
    // any order).
    const int chunk = blockIdx.x, bh = a.B * a.H - 1 - blockIdx.y, b = bh / a.H, h = bh % a.H;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub = lane / LPR, col = (lane % LPR) * 8;
    float cm[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) cm[e] = a.k_mean[(size_t)bh * D + col + e];
    const __nv_bfloat16 *kb = a.k + b * a.ks0 + h * a.ks1 + col;
    const int fr = chunk / a.cpf;
    const int r0 = fr * a.T + (chunk % a.cpf) * kRowsPerChunk;
    const int r1 = min((fr + 1) * a.T, r0 + kRowsPerChunk);
    constexpr int kStep = kStatsWarps * RPW;
    float rm2 = 0.f;
    for (int wbase = r0 + warp * RPW; wbase < r1; wbase += kStep * kUnroll2) {
        uint4 xk[kUnroll2];
        bool in[kUnroll2];
#pragma unroll
        for (int u = 0; u < kUnroll2; ++u) {
            const int r = wbase + sub + u * kStep;
            in[u] = r < r1;
            xk[u] = in[u] ? load16(kb + (long long)r * a.ks2) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kUnroll2; ++u) {
            float sq = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float t = elem8(xk[u], e) - cm[e];
                sq = fmaf(t, t, sq);
            }
            sq = row_sum<LPR>(sq);
            rm2 = in[u] ? fmaxf(rm2, sq) : rm2;   // rows past the chunk contribute nothing
        }
    }
    rm2 = warp_max(rm2);
    if (lane == 0) s_r[warp] = rm2;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int w = 0; w < kStatsWarps; ++w) m = fmaxf(m, s_r[w]);
        a.ws_rn2[(size_t)bh * a.nchunk + chunk] = m;
    }
}

__global__ void stats_finalize(StatsArgs a) {
    const int bh = blockIdx.x, lane = threadIdx.x;
    float r2 = 0.f, q2 = 0.f;
    for (int c = lane; c < a.nchunk; c += 32) {
        r2 = fmaxf(r2, a.ws_rn2[(size_t)bh * a.nchunk + c]);
        q2 = fmaxf(q2, a.ws_qn2[(size_t)bh * a.nchunk + c]);
    }
    r2 = warp_max(r2);
    q2 = warp_max(q2);
    if (lane == 0) {
        const float R = sqrtf(r2), Qm = sqrtf(q2);
        const float G = 2.0f * a.scale * Qm * R;
        a.k_rmax[bh] = R;
        a.q_nmax[bh] = Qm;
        a.gap[bh] = G;
        a.elig[bh] = (G <= a.tau) ? 1 : 0;
    }
}

int nchunks(int N) { return (N + kRowsPerChunk - 1) / kRowsPerChunk; }

// Per (b, h, segment of a plan): R over the key frames the segment's queries see
// and Qmax over the segment's query frames, from the frame-aligned chunk maxima.
__global__ void stats_segments(StatsArgs a, const int32_t *segments, int nseg, float *seg_rmax,
                               float *seg_gap, uint8_t *seg_elig) {
    const int bh = blockIdx.x;
    const float *rn2 = a.ws_rn2 + (size_t)bh * a.nchunk;
    const float *qn2 = a.ws_qn2 + (size_t)bh * a.nchunk;
    for (int sg = threadIdx.x; sg < nseg; sg += blockDim.x) {
        const int32_t *g = segments + kSegInts * sg;
        float r2 = 0.f, q2 = 0.f;
        for (int run = 0; run < 2; ++run)
            for (int f = g[2 + 2 * run] / a.T; f < g[3 + 2 * run] / a.T; ++f)
                for (int c = f * a.cpf; c < (f + 1) * a.cpf; ++c) r2 = fmaxf(r2, rn2[c]);
        for (int f = g[0] / a.T; f < (g[0] + g[1]) / a.T; ++f)
            for (int c = f * a.cpf; c < (f + 1) * a.cpf; ++c) q2 = fmaxf(q2, qn2[c]);
        const float R = sqrtf(r2), Qm = sqrtf(q2);
        const float G = 2.0f * a.scale * Qm * R;
        const size_t o = (size_t)bh * nseg + sg;
        seg_rmax[o] = R;
        seg_gap[o] = G;
        seg_elig[o] = (G <= a.tau) ? 1 : 0;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace vdit

using namespace vdit;

extern "C" size_t vdit_key_stats_workspace_size(int32_t B, int32_t H, int32_t N, int32_t D) {
    if (B < 1 || H < 1 || N < 1 || D < 1) return 0;
    const size_t slots = (size_t)B * H * nchunks(N);
    return slots * (size_t)(D + 2) * sizeof(float);
}

extern "C" vdit_status vdit_key_stats(const void *q, const void *k, int32_t B, int32_t H,
                                      int32_t N, int32_t D, const int64_t q_strides[3],
                                      const int64_t k_strides[3], float scale, float tau,
                                      float *k_mean, float *k_rmax, float *q_nmax,
                                      float *gap_bound, uint8_t *eligible, void *workspace,
                                      size_t workspace_bytes, void *stream) {
    clear_error();
    if (!q || !k || !q_strides || !k_strides || !k_mean || !k_rmax || !q_nmax || !gap_bound ||
        !eligible || !workspace) {
        set_error("vdit_key_stats: NULL pointer argument");
        return VDIT_ERR_INVALID;
    }
    if (B < 1 || H < 1 || N < 1) {
        set_error("vdit_key_stats: B=%d H=%d N=%d must be >= 1", B, H, N);
        return VDIT_ERR_INVALID;
    }
    if (D != 64 && D != 128) {
        set_error("vdit_key_stats: head dim D=%d not supported (64 or 128)", D);
        return VDIT_ERR_UNSUPPORTED;
    }
    for (int i = 0; i < 3; ++i) {
        if (q_strides[i] <= 0 || k_strides[i] <= 0 || q_strides[i] % 8 || k_strides[i] % 8) {
            set_error("vdit_key_stats: strides must be positive multiples of 8 elements");
            return VDIT_ERR_INVALID;
        }
    }
    if (!aligned16(q) || !aligned16(k)) {
        set_error("vdit_key_stats: q and k must be 16-byte aligned");
        return VDIT_ERR_INVALID;
    }
    const size_t need = vdit_key_stats_workspace_size(B, H, N, D);
    if (workspace_bytes < need) {
        set_error("vdit_key_stats: workspace of %zu bytes < %zu needed", workspace_bytes, need);
        return VDIT_ERR_INVALID;
    }
    if (!finite_positive(scale) || !(tau >= 0.f)) {
        set_error("vdit_key_stats: scale must be finite and > 0, tau >= 0");
        return VDIT_ERR_INVALID;
    }
    StatsArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.qs0 = q_strides[0]; a.qs1 = q_strides[1]; a.qs2 = q_strides[2];
    a.ks0 = k_strides[0]; a.ks1 = k_strides[1]; a.ks2 = k_strides[2];
    a.B = B; a.H = H; a.N = N; a.nchunk = nchunks(N);
    a.T = N; a.cpf = a.nchunk;
    a.scale = scale; a.tau = tau;
    const size_t slots = (size_t)B * H * a.nchunk;
    a.ws_colsum = static_cast<float *>(workspace);
    a.ws_qn2 = a.ws_colsum + slots * D;
    a.ws_rn2 = a.ws_qn2 + slots;
    a.k_mean = k_mean; a.k_rmax = k_rmax; a.q_nmax = q_nmax; a.gap = gap_bound;
    a.elig = eligible;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    dim3 grid(a.nchunk, B * H);
    if (D == 128) {
        stats_pass1<128><<<grid, kStatsThreads, 0, s>>>(a);
        stats_mean<<<B * H, 128, 0, s>>>(a, D);
        stats_pass2<128><<<grid, kStatsThreads, 0, s>>>(a);
    } else {
        stats_pass1<64><<<grid, kStatsThreads, 0, s>>>(a);
        stats_mean<<<B * H, 128, 0, s>>>(a, D);
        stats_pass2<64><<<grid, kStatsThreads, 0, s>>>(a);
    }
    stats_finalize<<<B * H, 32, 0, s>>>(a);
    VDIT_CUDA_TRY(cudaGetLastError());
    return VDIT_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of vdit_key_stats.
//
// Some callers cannot allocate device memory: a plugin whose host framework
// owns every device buffer through its own pool and forbids plugins from
// calling cudaMalloc, or a latency-critical loop that must not pay
// cudaMalloc's implicit device-wide synchronisation after start-up. This entry
// point runs the same three kernels as vdit_key_stats, but takes their scratch
// from a fixed array compiled into the library instead of from a caller buffer.
//
// The array below lives in device memory for as long as the library stays
// loaded, on every GPU that loads it. Every call shares it and it keeps the
// previous call's contents; the kernels overwrite every scratch slot they read
// (nothing needs to start at zero). Two calls whose kernels overlap on the GPU
// (e.g. on different streams, or on one device from several host threads
// without ordering) race on the array.
namespace vdit {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_key_stats_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the host-side symbol is only a stand-in, not a device address).
cudaError_t scratch_address(int device, void **out) {
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_scratch_addr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_key_stats_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return cudaSuccess;
}

}  // namespace
}  // namespace vdit

extern "C" vdit_status vdit_key_stats_noalloc(const void *q, const void *k, int32_t B, int32_t H,
                                              int32_t N, int32_t D, const int64_t q_strides[3],
                                              const int64_t k_strides[3], float scale, float tau,
                                              float *k_mean, float *k_rmax, float *q_nmax,
                                              float *gap_bound, uint8_t *eligible, void *stream) {
    clear_error();
    if (!q || !k || !q_strides || !k_strides || !k_mean || !k_rmax || !q_nmax || !gap_bound ||
        !eligible) {
        set_error("vdit_key_stats_noalloc: NULL pointer argument");
        return VDIT_ERR_INVALID;
    }
    if (B < 1 || H < 1 || N < 1) {
        set_error("vdit_key_stats_noalloc: B=%d H=%d N=%d must be >= 1", B, H, N);
        return VDIT_ERR_INVALID;
    }
    if (D != 64 && D != 128) {
        set_error("vdit_key_stats_noalloc: head dim D=%d not supported (64 or 128)", D);
        return VDIT_ERR_UNSUPPORTED;
    }
    for (int i = 0; i < 3; ++i) {
        if (q_strides[i] <= 0 || k_strides[i] <= 0 || q_strides[i] % 8 || k_strides[i] % 8) {
            set_error("vdit_key_stats_noalloc: strides must be positive multiples of 8 elements");
            return VDIT_ERR_INVALID;
        }
    }
    if (!aligned16(q) || !aligned16(k)) {
        set_error("vdit_key_stats_noalloc: q and k must be 16-byte aligned");
        return VDIT_ERR_INVALID;
    }
    if (!finite_positive(scale) || !(tau >= 0.f)) {
        set_error("vdit_key_stats_noalloc: scale must be finite and > 0, tau >= 0");
        return VDIT_ERR_INVALID;
    }
    const size_t need = vdit_key_stats_workspace_size(B, H, N, D);
    if (need > kNoAllocScratchBytes) {
        set_error("vdit_key_stats_noalloc: these sizes need %zu bytes of scratch, more than the "
                  "built-in %zu bytes (B*H*ceil(N/512)*(D+2)*4 must not exceed it); use "
                  "vdit_key_stats with a caller workspace", need, kNoAllocScratchBytes);
        return VDIT_ERR_INVALID;
    }
    int dev = -1;
    VDIT_CUDA_TRY(cudaGetDevice(&dev));
    void *scratch = nullptr;
    cudaError_t e = scratch_address(dev, &scratch);
    if (e != cudaSuccess) return cuda_fail(e, "vdit_key_stats_noalloc: cudaGetSymbolAddress");
    StatsArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.qs0 = q_strides[0]; a.qs1 = q_strides[1]; a.qs2 = q_strides[2];
    a.ks0 = k_strides[0]; a.ks1 = k_strides[1]; a.ks2 = k_strides[2];
    a.B = B; a.H = H; a.N = N; a.nchunk = nchunks(N);
    a.T = N; a.cpf = a.nchunk;
    a.scale = scale; a.tau = tau;
    const size_t slots = (size_t)B * H * a.nchunk;
    a.ws_colsum = static_cast<float *>(scratch);
    a.ws_qn2 = a.ws_colsum + slots * D;
    a.ws_rn2 = a.ws_qn2 + slots;
    a.k_mean = k_mean; a.k_rmax = k_rmax; a.q_nmax = q_nmax; a.gap = gap_bound;
    a.elig = eligible;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    dim3 grid(a.nchunk, B * H);
    if (D == 128) {
        stats_pass1<128><<<grid, kStatsThreads, 0, s>>>(a);
        stats_mean<<<B * H, 128, 0, s>>>(a, D);
        stats_pass2<128><<<grid, kStatsThreads, 0, s>>>(a);
    } else {
        stats_pass1<64><<<grid, kStatsThreads, 0, s>>>(a);
        stats_mean<<<B * H, 128, 0, s>>>(a, D);
        stats_pass2<64><<<grid, kStatsThreads, 0, s>>>(a);
    }
    stats_finalize<<<B * H, 32, 0, s>>>(a);
    VDIT_CUDA_TRY(cudaGetLastError());
    return VDIT_OK;
}

extern "C" size_t vdit_key_stats_framed_workspace_size(const vdit_plan *plan, int32_t B, int32_t H,
                                                       int32_t D) {
    if (!plan || B < 1 || H < 1 || D < 1) return 0;
    const size_t slots = (size_t)B * H * plan->F * nchunks(plan->T);
    return slots * (size_t)(D + 2) * sizeof(float);
}

extern "C" vdit_status vdit_key_stats_framed(const vdit_plan *plan, const void *q, const void *k,
                                             int32_t B, int32_t H, int32_t D,
                                             const int64_t q_strides[3], const int64_t k_strides[3],
                                             float scale, float tau, float *k_mean, float *seg_rmax,
                                             float *seg_gap, uint8_t *seg_eligible, void *workspace,
                                             size_t workspace_bytes, void *stream) {
    clear_error();
    if (!plan || !q || !k || !q_strides || !k_strides || !k_mean || !seg_rmax || !seg_gap ||
        !seg_eligible || !workspace) {
        set_error("vdit_key_stats_framed: NULL pointer argument");
        return VDIT_ERR_INVALID;
    }
    if (B < 1 || H < 1) {
        set_error("vdit_key_stats_framed: B=%d H=%d must be >= 1", B, H);
        return VDIT_ERR_INVALID;
    }
    if (D != 64 && D != 128) {
        set_error("vdit_key_stats_framed: head dim D=%d not supported (64 or 128)", D);
        return VDIT_ERR_UNSUPPORTED;
    }
    for (int i = 0; i < 3; ++i) {
        if (q_strides[i] <= 0 || k_strides[i] <= 0 || q_strides[i] % 8 || k_strides[i] % 8) {
            set_error("vdit_key_stats_framed: strides must be positive multiples of 8 elements");
            return VDIT_ERR_INVALID;
        }
    }
    if (!aligned16(q) || !aligned16(k)) {
        set_error("vdit_key_stats_framed: q and k must be 16-byte aligned");
        return VDIT_ERR_INVALID;
    }
    const size_t need = vdit_key_stats_framed_workspace_size(plan, B, H, D);
    if (workspace_bytes < need) {
        set_error("vdit_key_stats_framed: workspace of %zu bytes < %zu needed", workspace_bytes, need);
        return VDIT_ERR_INVALID;
    }
    if (!finite_positive(scale) || !(tau >= 0.f)) {
        set_error("vdit_key_stats_framed: scale must be finite and > 0, tau >= 0");
        return VDIT_ERR_INVALID;
    }
    int dev = -1;
    VDIT_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != plan->device) {
        set_error("vdit_key_stats_framed: plan was built on device %d, current device is %d",
                  plan->device, dev);
        return VDIT_ERR_INVALID;
    }
    StatsArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.qs0 = q_strides[0]; a.qs1 = q_strides[1]; a.qs2 = q_strides[2];
    a.ks0 = k_strides[0]; a.ks1 = k_strides[1]; a.ks2 = k_strides[2];
    a.B = B; a.H = H; a.N = (int)plan->N;
    a.T = plan->T; a.cpf = nchunks(plan->T); a.nchunk = plan->F * a.cpf;
    a.scale = scale; a.tau = tau;
    const size_t slots = (size_t)B * H * a.nchunk;
    a.ws_colsum = static_cast<float *>(workspace);
    a.ws_qn2 = a.ws_colsum + slots * D;
    a.ws_rn2 = a.ws_qn2 + slots;
    a.k_mean = k_mean; a.k_rmax = nullptr; a.q_nmax = nullptr; a.gap = nullptr; a.elig = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    dim3 grid(a.nchunk, B * H);
    if (D == 128) {
        stats_pass1<128><<<grid, kStatsThreads, 0, s>>>(a);
        stats_mean<<<B * H, 128, 0, s>>>(a, D);
        stats_pass2<128><<<grid, kStatsThreads, 0, s>>>(a);
    } else {
        stats_pass1<64><<<grid, kStatsThreads, 0, s>>>(a);
        stats_mean<<<B * H, 128, 0, s>>>(a, D);
        stats_pass2<64><<<grid, kStatsThreads, 0, s>>>(a);
    }
    stats_segments<<<B * H, 64, 0, s>>>(a, plan->d_segments, plan->h.n_segments, seg_rmax, seg_gap,
                                         seg_eligible);
    VDIT_CUDA_TRY(cudaGetLastError());
    return VDIT_OK;
}

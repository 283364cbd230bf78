// Head-group pipelining of attention over host-resident Q, K, V, O.
//
// "HeyGen x Google Cloud: Bringing Avatar IV to TPUs", "Hiding the Collective"
// (Fig. 2): the all-to-all that brings each device its heads sat uncovered on
// the critical path; splitting the heads into independent groups, each with
// its own transfer -> attention -> transfer chain, lets every middle transfer
// hide behind another group's attention, leaving only the first transfer in
// and the last transfer out exposed. Splitting by heads leaves the token order
// (and so the frame-window mask) untouched: each group gets the same mask as one launch
// over all heads.
//
// On one GB300 the wire is the host link: Q, K, V of head group g are copied
// in on one stream, the group's key statistics and attention run on the
// compute stream of its slot, and its O (and LSE) are copied out on another
// stream. Two device slots alternate, so group g+1's copy-in and group g-1's
// copy-out overlap group g's kernels, and group g+1's kernels can fill the
// SMs that group g's last wave leaves idle. Events order the streams; nothing
// waits on the host. Groups may have different sizes: small first and last
// groups shorten the exposed first copy-in and last copy-out.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "vdit_internal.h"

namespace {

constexpr int kSlots = 2;

struct Slot {
    uint8_t *q = nullptr, *k = nullptr, *v = nullptr, *o = nullptr;
    float *lse = nullptr;
    float *k_mean = nullptr, *k_rmax = nullptr, *q_nmax = nullptr, *gap = nullptr;
    uint8_t *elig = nullptr;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    // qk_ready: q and k landed (the key statistics may start); in_ready: v too
    cudaEvent_t qk_ready = nullptr, in_ready = nullptr, computed = nullptr, out_done = nullptr;
};

size_t align_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Default group schedule: 1, 2, ..., c-1 heads, then groups of c, then c-1, ...,
// 1, with c = 4. The first group's copy-in and the last group's copy-out are
// the only transfers left exposed, so they are the smallest; each later copy-in
// (about 0.6 of a head's attention time per head on the host link of a GB300)
// still hides behind the previous, smaller group's kernels. Heads beyond the
// ramps that do not fill a group of c are spread over the middle groups, one
// more per group in turn (a group takes several when there are fewer middle
// groups than leftover heads).
// Returns the group count (sizes in out[]), or 0 when H is too small for the
// ramps (the caller then splits evenly into groups of about c).
constexpr int kTaperCap = 4;
int tapered_split(int H, int *out) {
    const int ramp = kTaperCap * (kTaperCap - 1) / 2;   // 1 + ... + (c-1)
    if (H < 2 * ramp + kTaperCap) return 0;
    const int mid = H - 2 * ramp, nmid = mid / kTaperCap, extra = mid % kTaperCap;
    if (2 * (kTaperCap - 1) + nmid > 64) return 0;
    // nmid >= 1 here, since mid >= c
    const int each = kTaperCap + extra / nmid, rest = extra % nmid;
    int g = 0;
    for (int i = 1; i < kTaperCap; ++i) out[g++] = i;
    for (int i = 0; i < nmid; ++i) out[g++] = each + (i < rest ? 1 : 0);
    for (int i = kTaperCap - 1; i >= 1; --i) out[g++] = i;
    return g;
}

}  // namespace

// The schedule vdit_pipeline_create picks for groups = 0: the tapered split when
// H allows the ramps, else ceil(H / c) groups of equal size (the last may be
// smaller), by the same rules as the create call below.
extern "C" int32_t vdit_pipeline_default_groups(int32_t H, int32_t *out, int32_t cap) {
    if (H < 1 || !out || cap < 1) return 0;
    int taper[64];
    int n = tapered_split(H, taper);
    if (n > 0) {
        if (n > cap) return 0;
        for (int i = 0; i < n; ++i) out[i] = taper[i];
        return n;
    }
    const int groups = (H + kTaperCap - 1) / kTaperCap, hg = (H + groups - 1) / groups;
    n = (H + hg - 1) / hg;
    if (n > cap) return 0;
    for (int i = 0; i < n; ++i) out[i] = (i + 1) * hg <= H ? hg : H - i * hg;
    return n;
}

struct vdit_pipeline {
    const vdit_plan *plan = nullptr;
    int B = 0, H = 0, D = 0, N = 0, groups = 0, hg = 0, device = -1;
    int *first = nullptr;    // first head of each group, groups + 1 entries
    void *mem = nullptr;
    Slot slot[kSlots];
    cudaStream_t s_in = nullptr, s_out = nullptr, s_cmp[kSlots] = {};
    cudaEvent_t start = nullptr;
    cudaEvent_t join[2 + kSlots] = {};   // error path: the caller's stream waits for every internal stream
};

namespace {

void release(vdit_pipeline *p) {
    if (!p) return;
    for (Slot &s : p->slot) {
        if (s.qk_ready) cudaEventDestroy(s.qk_ready);
        if (s.in_ready) cudaEventDestroy(s.in_ready);
        if (s.computed) cudaEventDestroy(s.computed);
        if (s.out_done) cudaEventDestroy(s.out_done);
    }
    if (p->start) cudaEventDestroy(p->start);
    for (cudaEvent_t e : p->join)
        if (e) cudaEventDestroy(e);
    if (p->s_in) cudaStreamDestroy(p->s_in);
    for (cudaStream_t s : p->s_cmp)
        if (s) cudaStreamDestroy(s);
    if (p->s_out) cudaStreamDestroy(p->s_out);
    if (p->mem) cudaFree(p->mem);
    delete[] p->first;
    delete p;
}

// Layout of one head group's tensor on the device, chosen from the host layout
// so that each (batch, tensor) moves in as few copies as possible:
//   token-major host (heads adjacent inside a token row): device [n][hc][D],
//     one 2-D copy of N rows x hc*D elements per batch;
//   otherwise: device [hc][n][D], one copy per head (1-D when the head's rows
//     are contiguous on the host).
struct GroupLayout {
    bool token_major;
    int64_t dev_strides[3];  // elements, for (b, h, n)
};

GroupLayout group_layout(const int64_t hs[3], int N, int D, int hc) {
    GroupLayout L;
    L.token_major = hs[1] == D && hs[2] >= (int64_t)hc * D;
    if (L.token_major) {
        L.dev_strides[0] = (int64_t)N * hc * D;
        L.dev_strides[1] = D;
        L.dev_strides[2] = (int64_t)hc * D;
    } else {
        L.dev_strides[0] = (int64_t)hc * N * D;
        L.dev_strides[1] = (int64_t)N * D;
        L.dev_strides[2] = D;
    }
    return L;
}

// Copy heads [h0, h0 + hc) of every batch between a host tensor (element
// strides hs for b, h, n; d contiguous) and a dense device group buffer.
// `elem` is the element size; `dir` is cudaMemcpyHostToDevice or DeviceToHost.
cudaError_t copy_group(uint8_t *dev, uint8_t *host, const int64_t hs[3], int B, int N, int D, int h0,
                       int hc, size_t elem, cudaMemcpyKind dir, cudaStream_t s) {
    const GroupLayout L = group_layout(hs, N, D, hc);
    for (int b = 0; b < B; ++b) {
        uint8_t *hb = host + ((int64_t)b * hs[0] + (int64_t)h0 * hs[1]) * elem;
        uint8_t *db = dev + (int64_t)b * L.dev_strides[0] * elem;
        if (L.token_major) {
            const size_t width = (size_t)hc * D * elem, hpitch = (size_t)hs[2] * elem;
            cudaError_t e = dir == cudaMemcpyHostToDevice
                                ? cudaMemcpy2DAsync(db, width, hb, hpitch, width, N, dir, s)
                                : cudaMemcpy2DAsync(hb, hpitch, db, width, width, N, dir, s);
            if (e != cudaSuccess) return e;
            continue;
        }
        for (int h = 0; h < hc; ++h) {
            uint8_t *hh = hb + (int64_t)h * hs[1] * elem;
            uint8_t *dh = db + (int64_t)h * L.dev_strides[1] * elem;
            const size_t row = (size_t)D * elem, hpitch = (size_t)hs[2] * elem;
            cudaError_t e;
            if (hs[2] == D) {   // the head's N rows are contiguous
                e = dir == cudaMemcpyHostToDevice ? cudaMemcpyAsync(dh, hh, row * N, dir, s)
                                                  : cudaMemcpyAsync(hh, dh, row * N, dir, s);
            } else {
                e = dir == cudaMemcpyHostToDevice ? cudaMemcpy2DAsync(dh, row, hh, hpitch, row, N, dir, s)
                                                  : cudaMemcpy2DAsync(hh, hpitch, dh, row, row, N, dir, s);
            }
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace

using namespace vdit;

extern "C" vdit_status vdit_pipeline_create(const vdit_plan *plan, int32_t B, int32_t H, int32_t D,
                                            int32_t groups, const int32_t *group_heads,
                                            vdit_pipeline **out) {
    clear_error();
    if (!out) { set_error("vdit_pipeline_create: out is NULL"); return VDIT_ERR_INVALID; }
    *out = nullptr;
    if (!plan) { set_error("vdit_pipeline_create: plan is NULL"); return VDIT_ERR_INVALID; }
    if (B < 1 || H < 1) { set_error("vdit_pipeline_create: B=%d H=%d must be >= 1", B, H); return VDIT_ERR_INVALID; }
    if (D != 64 && D != 128) {
        set_error("vdit_pipeline_create: head dim D=%d not supported (64 or 128)", D);
        return VDIT_ERR_UNSUPPORTED;
    }
    if (groups < 0 || groups > H || (groups == 0 && group_heads)) {
        set_error("vdit_pipeline_create: groups=%d must be in [1, H=%d] (or 0, without group_heads)", groups, H);
        return VDIT_ERR_INVALID;
    }
    if (group_heads) {
        long long sum = 0;
        for (int g = 0; g < groups; ++g) {
            if (group_heads[g] < 1) {
                set_error("vdit_pipeline_create: group_heads[%d]=%d must be >= 1", g, group_heads[g]);
                return VDIT_ERR_INVALID;
            }
            sum += group_heads[g];
        }
        if (sum != H) {
            set_error("vdit_pipeline_create: group_heads sum to %lld, not H=%d", sum, H);
            return VDIT_ERR_INVALID;
        }
    }
    int dev = -1;
    VDIT_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != plan->device) {
        set_error("vdit_pipeline_create: plan was built on device %d, current device is %d", plan->device, dev);
        return VDIT_ERR_INVALID;
    }
    vdit_pipeline *p = new (std::nothrow) vdit_pipeline();
    if (!p) { set_error("vdit_pipeline_create: out of host memory"); return VDIT_ERR_NOMEM; }
    p->plan = plan;
    p->B = B; p->H = H; p->D = D; p->N = (int)plan->N; p->device = dev;
    int taper[64];
    if (groups == 0) {
        groups = tapered_split(H, taper);
        if (groups > 0) group_heads = taper;
        else groups = (H + kTaperCap - 1) / kTaperCap;
    }
    p->first = new (std::nothrow) int[groups + 1];
    if (!p->first) { release(p); set_error("vdit_pipeline_create: out of host memory"); return VDIT_ERR_NOMEM; }
    if (group_heads) {
        p->groups = groups;
        p->first[0] = 0;
        p->hg = 0;
        for (int g = 0; g < groups; ++g) {
            p->first[g + 1] = p->first[g] + group_heads[g];
            if (group_heads[g] > p->hg) p->hg = group_heads[g];
        }
    } else {   // equal split of ceil(H / groups) heads, no empty trailing group
        p->hg = (H + groups - 1) / groups;
        p->groups = (H + p->hg - 1) / p->hg;
        for (int g = 0; g <= p->groups; ++g) p->first[g] = g * p->hg < H ? g * p->hg : H;
    }
    if (p->first[p->groups] != H) {   // every schedule above covers the H heads exactly
        const int covered = p->first[p->groups];
        release(p);
        set_error("vdit_pipeline_create: head groups cover %d of %d heads", covered, H);
        return VDIT_ERR_INVALID;
    }
    const size_t N = (size_t)p->N, hg = (size_t)p->hg;
    const size_t t_bytes = align_up((size_t)B * hg * N * D * 2);
    const size_t lse_bytes = align_up((size_t)B * hg * N * 4);
    const size_t stat_bytes = align_up((size_t)B * hg * D * 4) + 3 * align_up((size_t)B * hg * 4) +
                              align_up((size_t)B * hg);
    const size_t ws_bytes = align_up(vdit_key_stats_workspace_size(B, p->hg, p->N, D));
    const size_t per_slot = 4 * t_bytes + lse_bytes + stat_bytes + ws_bytes;
    cudaError_t e = device_alloc(&p->mem, per_slot * kSlots);
    if (e != cudaSuccess) {
        release(p);
        set_error("vdit_pipeline_create: device allocation of %zu bytes failed (%s)", per_slot * kSlots,
                  cudaGetErrorString(e));
        return VDIT_ERR_NOMEM;
    }
    for (int i = 0; i < kSlots; ++i) {
        uint8_t *m = static_cast<uint8_t *>(p->mem) + i * per_slot;
        Slot &s = p->slot[i];
        s.q = m; m += t_bytes;
        s.k = m; m += t_bytes;
        s.v = m; m += t_bytes;
        s.o = m; m += t_bytes;
        s.lse = reinterpret_cast<float *>(m); m += lse_bytes;
        s.k_mean = reinterpret_cast<float *>(m); m += align_up((size_t)B * hg * D * 4);
        s.k_rmax = reinterpret_cast<float *>(m); m += align_up((size_t)B * hg * 4);
        s.q_nmax = reinterpret_cast<float *>(m); m += align_up((size_t)B * hg * 4);
        s.gap = reinterpret_cast<float *>(m); m += align_up((size_t)B * hg * 4);
        s.elig = m; m += align_up((size_t)B * hg);
        s.ws = m; s.ws_bytes = ws_bytes;
        for (cudaEvent_t *ev : {&s.qk_ready, &s.in_ready, &s.computed, &s.out_done}) {
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) {
                release(p);
                return cuda_fail(e, "vdit_pipeline_create: cudaEventCreate");
            }
        }
    }
    for (cudaEvent_t &j : p->join)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&j, cudaEventDisableTiming);
    if (e == cudaSuccess && (e = cudaEventCreateWithFlags(&p->start, cudaEventDisableTiming)) == cudaSuccess &&
        (e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking)) == cudaSuccess)
        e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i)
        e = cudaStreamCreateWithFlags(&p->s_cmp[i], cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        release(p);
        return cuda_fail(e, "vdit_pipeline_create: stream/event creation");
    }
    *out = p;
    return VDIT_OK;
}

namespace {

// Queues every head group of one run (see vdit_pipeline_run). Returns at the
// first error; what was queued before it stays queued.
vdit_status enqueue_groups(vdit_pipeline *p, const void *q_host, const void *k_host, const void *v_host,
                           void *o_host, float *lse_host, const int64_t host_strides[3], float scale,
                           float tau, int32_t mode, cudaStream_t caller) {
    VDIT_CUDA_TRY(cudaEventRecord(p->start, caller));
    VDIT_CUDA_TRY(cudaStreamWaitEvent(p->s_in, p->start, 0));
    for (cudaStream_t sc : p->s_cmp) VDIT_CUDA_TRY(cudaStreamWaitEvent(sc, p->start, 0));
    VDIT_CUDA_TRY(cudaStreamWaitEvent(p->s_out, p->start, 0));
    // A previous run may have been queued on another stream: the first groups of
    // this run reuse its slots only after its kernels and copies of those slots
    // are done (on one stream the start event already orders this; an event never
    // recorded is a wait that completes at once).
    for (int i = 0; i < kSlots; ++i) {
        VDIT_CUDA_TRY(cudaStreamWaitEvent(p->s_in, p->slot[i].computed, 0));
        VDIT_CUDA_TRY(cudaStreamWaitEvent(p->s_cmp[i], p->slot[i].out_done, 0));
    }
    const int B = p->B, N = p->N, D = p->D, H = p->H;
    for (int g = 0; g < p->groups; ++g) {
        const int h0 = p->first[g], hc = p->first[g + 1] - h0;
        Slot &s = p->slot[g % kSlots];
        cudaStream_t s_cmp = p->s_cmp[g % kSlots];
        const bool reuse = g >= kSlots;
        const GroupLayout L = group_layout(host_strides, N, D, hc);
        // copy in: the slot's inputs are free once group g - 2's kernels finished
        if (reuse) VDIT_CUDA_TRY(cudaStreamWaitEvent(p->s_in, s.computed, 0));
        const void *ins[3] = {q_host, k_host, v_host};
        uint8_t *dsts[3] = {s.q, s.k, s.v};
        for (int t = 0; t < 3; ++t) {
            VDIT_CUDA_TRY(copy_group(dsts[t], static_cast<uint8_t *>(const_cast<void *>(ins[t])), host_strides, B,
                                     N, D, h0, hc, 2, cudaMemcpyHostToDevice, p->s_in));
            if (t == 1) VDIT_CUDA_TRY(cudaEventRecord(s.qk_ready, p->s_in));
        }
        VDIT_CUDA_TRY(cudaEventRecord(s.in_ready, p->s_in));
        // kernels: the slot's O is free once group g - 2's copy-out finished. The key
        // statistics read only q and k, so they start while v is still copying.
        VDIT_CUDA_TRY(cudaStreamWaitEvent(s_cmp, s.qk_ready, 0));
        if (reuse) VDIT_CUDA_TRY(cudaStreamWaitEvent(s_cmp, s.out_done, 0));
        vdit_status st = vdit_key_stats(s.q, s.k, B, hc, N, D, L.dev_strides, L.dev_strides, scale, tau,
                                        s.k_mean, s.k_rmax, s.q_nmax, s.gap, s.elig, s.ws, s.ws_bytes,
                                        s_cmp);
        if (st != VDIT_OK) return st;
        VDIT_CUDA_TRY(cudaStreamWaitEvent(s_cmp, s.in_ready, 0));
        st = vdit_attn_fwd(p->plan, s.q, s.k, s.v, s.o, VDIT_O_BF16, lse_host ? s.lse : nullptr, B, hc, D,
                           L.dev_strides, L.dev_strides, L.dev_strides, L.dev_strides, scale, s.k_mean,
                           s.k_rmax, s.elig, mode, s_cmp);
        if (st != VDIT_OK) return st;
        VDIT_CUDA_TRY(cudaEventRecord(s.computed, s_cmp));
        // copy out
        VDIT_CUDA_TRY(cudaStreamWaitEvent(p->s_out, s.computed, 0));
        VDIT_CUDA_TRY(copy_group(s.o, static_cast<uint8_t *>(o_host), host_strides, B, N, D, h0, hc, 2,
                                 cudaMemcpyDeviceToHost, p->s_out));
        if (lse_host) {
            // lse: host [B, H, N] dense, device [B, hc, N]
            for (int b = 0; b < B; ++b)
                VDIT_CUDA_TRY(cudaMemcpyAsync(lse_host + ((int64_t)b * H + h0) * N, s.lse + (int64_t)b * hc * N,
                                              (size_t)hc * N * sizeof(float), cudaMemcpyDeviceToHost, p->s_out));
        }
        VDIT_CUDA_TRY(cudaEventRecord(s.out_done, p->s_out));
    }
    // the caller's stream continues once every group's output has landed
    for (int i = 0; i < kSlots && i < p->groups; ++i)
        VDIT_CUDA_TRY(cudaStreamWaitEvent(caller, p->slot[i].out_done, 0));
    return VDIT_OK;
}

}  // namespace

extern "C" vdit_status vdit_pipeline_run(vdit_pipeline *p, const void *q_host, const void *k_host,
                                         const void *v_host, void *o_host, float *lse_host,
                                         const int64_t host_strides[3], float scale, float tau,
                                         int32_t mode, void *stream) {
    clear_error();
    if (!p) { set_error("vdit_pipeline_run: pipeline is NULL"); return VDIT_ERR_INVALID; }
    if (!q_host || !k_host || !v_host || !o_host || !host_strides) {
        set_error("vdit_pipeline_run: NULL pointer argument");
        return VDIT_ERR_INVALID;
    }
    for (int i = 0; i < 3; ++i)
        if (host_strides[i] <= 0) {
            set_error("vdit_pipeline_run: host strides must be positive");
            return VDIT_ERR_INVALID;
        }
    if (host_strides[2] < p->D) {
        set_error("vdit_pipeline_run: host token stride is below D");
        return VDIT_ERR_INVALID;
    }
    // checked here too, before any copy is queued (the per-group calls repeat them)
    if (!finite_positive(scale) || !(tau >= 0.f)) {
        set_error("vdit_pipeline_run: scale must be finite and > 0, tau >= 0");
        return VDIT_ERR_INVALID;
    }
    if (mode < VDIT_MODE_AUTO || mode > VDIT_MODE_FORCE_STATIC) {
        set_error("vdit_pipeline_run: mode=%d invalid", mode);
        return VDIT_ERR_INVALID;
    }
    int dev = -1;
    VDIT_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != p->device) {
        set_error("vdit_pipeline_run: pipeline was created on device %d, current device is %d", p->device, dev);
        return VDIT_ERR_INVALID;
    }
    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    const vdit_status st = enqueue_groups(p, q_host, k_host, v_host, o_host, lse_host, host_strides, scale,
                                          tau, mode, caller);
    if (st != VDIT_OK) {
        // Copies and kernels of earlier groups may still be queued on the internal
        // streams: the caller's stream waits for all of them, so that synchronising
        // it still covers every access to the host buffers.
        cudaStream_t ss[2 + kSlots] = {p->s_in, p->s_out};
        for (int i = 0; i < kSlots; ++i) ss[2 + i] = p->s_cmp[i];
        for (int i = 0; i < 2 + kSlots; ++i)
            if (cudaEventRecord(p->join[i], ss[i]) == cudaSuccess) cudaStreamWaitEvent(caller, p->join[i], 0);
    }
    return st;
}

extern "C" void vdit_pipeline_destroy(vdit_pipeline *p) {
    if (!p) return;
    cudaStreamSynchronize(p->s_in);
    for (cudaStream_t sc : p->s_cmp) cudaStreamSynchronize(sc);
    cudaStreamSynchronize(p->s_out);
    release(p);
}

/*
 * vdit.h -- C ABI of libvdit: frame-window + reference-frame block-sparse
 * self-attention for video diffusion transformers, hand-written for sm_103a.
 *
 * The operation is the sparse attention of the super-resolution stage described in
 * "HeyGen x Google Cloud: Bringing Avatar IV to TPUs":
 *   - "Deleting the Mask" (Fig. 3): every query in frame f attends to the keys
 *     of frames g with |f - g| <= W, plus one global reference frame. Blocks
 *     whose size is a multiple of 16 and divides the frame's token span are
 *     entirely live or entirely dead, so one pass needs no mask predicate, no
 *     padding and no second pass for the reference frame.
 *   - "Unchaining the Softmax" (Fig. 4): the running max of online softmax is
 *     replaced by a precomputed per-row upper bound on the logits,
 *     scale * (q . c + |q| * max_j |k_j - c|), with c the per-head key mean;
 *     a head with a loose bound runs online softmax instead, in the same
 *     kernel.
 *   - "Proving the Pixels Didn't Change": the final P.V product runs in bf16.
 *
 * Conventions shared by every call:
 *   - Tensors Q, K, V, O are [B, H, N, D] with the last dimension contiguous.
 *     Strides are given in ELEMENTS for (b, h, n), as int64_t[3]. Base
 *     addresses must be 16-byte aligned and the three strides multiples of
 *     16 bytes (TMA requirement). N = num_frames * tokens_per_frame, tokens
 *     frame-major. D is 64 or 128.
 *   - Every tensor argument is caller-owned DEVICE memory; the library never
 *     frees it. A plan owns only its own device buffers.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Every call is asynchronous on that stream, except vdit_attn_plan and
 *     vdit_plan_status, which synchronise it once.
 *   - Arguments are checked on the host before any launch. On error the call
 *     launches nothing, returns a non-zero vdit_status and sets a thread-local
 *     message readable through vdit_last_error().
 */
#ifndef VDIT_H
#define VDIT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VDIT_API __attribute__((visibility("default")))
#else
#define VDIT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VDIT_OK = 0,
    VDIT_ERR_INVALID = 1,     /* bad argument: shape, stride, alignment, null pointer */
    VDIT_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. D not in {64,128}) */
    VDIT_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    VDIT_ERR_NOMEM = 4,       /* device allocation for a plan failed */
    VDIT_ERR_TIMEOUT = 5      /* a kernel's bounded wait expired (see vdit_plan_status) */
} vdit_status;

enum { VDIT_O_BF16 = 0, VDIT_O_F32 = 1 };
enum { VDIT_MODE_AUTO = 0, VDIT_MODE_FORCE_ONLINE = 1, VDIT_MODE_FORCE_STATIC = 2 };
/* Which part of the mask a plan schedules (vdit_attn_plan_part). */
enum { VDIT_PART_ALL = 0, VDIT_PART_WINDOW = 1, VDIT_PART_REFERENCE = 2 };
/* Tiling of the two-pass ablation (vdit_attn_fwd_two_pass). */
enum { VDIT_TILES_FRAME = 0, VDIT_TILES_128 = 1 };

typedef struct vdit_plan vdit_plan; /* opaque, owned by the library */

/* Read-only view of a plan. All d_* pointers are device memory owned by the
 * plan and valid until vdit_plan_destroy. Counts are per (b, h) head. */
typedef struct {
    int32_t num_frames, tokens_per_frame, window_radius, ref_frame, block_size;
    int32_t dense;          /* 1 when every query sees every key (W >= F-1) */
    int64_t num_tokens;     /* N = F * T */
    int32_t n_qblocks;      /* ceil(N / block_size) */
    int64_t nnz;            /* live (query block, key block) pairs */
    int64_t live_pairs;     /* live (query token, key token) pairs */
    int32_t n_segments;     /* groups of consecutive frames sharing one key-run list */
    int32_t n_units;        /* attention work units per head (pairs of 128-row query tiles) */
    int32_t n_classes;      /* cost classes of the units (longest first) */
    const int32_t *d_row_ptr;    /* [n_qblocks + 1] CSR row offsets */
    const int32_t *d_col_idx;    /* [nnz] live key blocks, ascending per row */
    const int32_t *d_frame_runs; /* [F][4]: lo0, hi0, lo1, hi1 key tokens; (0,0) = no 2nd run */
    const int32_t *d_segments;   /* [n_segments][8]: row0, rows, lo0, hi0, lo1, hi1, ntiles, keys;
                                    ntiles = ceil(rows / 128), or floor when the segment's
                                    last rows % 128 rows went to a gathered tile */
    const int32_t *d_units;      /* [n_units]: (segment << 16) | tile pair, longest first */
    const int32_t *d_class_off;  /* [n_classes + 1] unit offsets of the cost classes */
    int32_t part;                /* VDIT_PART_*: the part of the mask this plan schedules */
    int32_t n_gathers;           /* query tiles per head that vdit_attn_fwd runs in a second
                                    launch: gathered tiles, which hold the ragged last rows
                                    (rows % 128, a multiple of 16 up to 64) of two to eight
                                    segments of at least 1024 rows each and visit the union
                                    of their key runs (at most two runs, at least a quarter
                                    fewer keys than the tails would visit apart), masking
                                    each row to its own runs; or, in a plan without those and
                                    with at least 32 tile pairs per head, tail tiles: the
                                    tiles of the last 8 pairs of the last segment in unit
                                    order, one record (one piece: the rows the tile owns)
                                    each, no longer in d_units */
    const int32_t *d_gathers;    /* [n_gathers][32]: pieces, rows, lo0, hi0, lo1, hi1 (the
                                    union), 1, keys, then per piece: segment, first row, rows */
} vdit_plan_info;

/* Build the block schedule of the frame-window + reference-frame mask
 * ("Deleting the Mask", Fig. 3).
 *   num_frames F >= 1, tokens_per_frame T >= 1, window_radius W >= 0,
 *   ref_frame in [-1, F-1] (-1 = no reference frame),
 *   block_size bs: a multiple of 16; it must divide T unless the mask is dense
 *   (W >= F-1), where a ragged last block is allowed. F*T < 2^31.
 * Allocates the plan's device buffers, launches the schedule kernels on
 * `stream`, and synchronises once to read the counts. *out receives the plan
 * (NULL on error). Errors: VDIT_ERR_INVALID (argument, or a CSR with 2^31 or
 * more live blocks), VDIT_ERR_UNSUPPORTED (a segment -- consecutive frames
 * sharing one key-run list, the whole sequence when dense -- of more than
 * 2^24 query rows: its 128-row tile pairs would not fit the 16-bit pair field
 * of d_units), VDIT_ERR_NOMEM, VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_attn_plan(int32_t num_frames, int32_t tokens_per_frame, int32_t window_radius,
                           int32_t ref_frame, int32_t block_size, void *stream, vdit_plan **out);

/* A plan for one part of the mask, for the two-pass form of the attention that
 * "Deleting the Mask" describes as the design before frame alignment: the
 * frame window and the reference frame run as two separate attention passes
 * whose results a merge pass combines (vdit_attn_fwd_two_pass).
 *   part = VDIT_PART_ALL: the whole mask, exactly vdit_attn_plan;
 *   part = VDIT_PART_WINDOW: the frames g with |f - g| <= W only;
 *   part = VDIT_PART_REFERENCE: the reference frame only, for query frames whose
 *     window does not contain it (the other frames see no key and get no work).
 * The two parts partition every query's live keys. Arguments and errors as
 * vdit_attn_plan; the window and reference parts also need a reference frame
 * (ref >= 0) and a window that does not cover every frame (W < F-1), else
 * VDIT_ERR_INVALID. */
VDIT_API vdit_status vdit_attn_plan_part(int32_t num_frames, int32_t tokens_per_frame,
                                         int32_t window_radius, int32_t ref_frame, int32_t block_size,
                                         int32_t part, void *stream, vdit_plan **out);

/* Re-launch the schedule kernels into the plan's existing buffers on `stream`
 * (asynchronous, no allocation, no synchronisation). The contents equal those
 * written by vdit_attn_plan. Errors: VDIT_ERR_INVALID (null plan), VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_plan_rebuild(vdit_plan *plan, void *stream);

/* Fill *info with the plan's counts and device pointers. */
VDIT_API vdit_status vdit_plan_get_info(const vdit_plan *plan, vdit_plan_info *info);

/* Synchronise `stream`, then report and clear the plan's device status word,
 * which a kernel launched with this plan sets when one of its bounded waits
 * expires. *code receives the raw word (0 = none). Returns VDIT_OK when the
 * word was 0, VDIT_ERR_TIMEOUT otherwise. */
VDIT_API vdit_status vdit_plan_status(vdit_plan *plan, void *stream, int32_t *code);

/* Block census of the plan's whole mask (all parts, whatever part the plan
 * schedules) under a tiling that ignores frames
 * ("Deleting the Mask": tiles of a multiple of 128 tokens straddle frame
 * boundaries, and about one live block in five comes out partial). Over the
 * N x N token pairs cut into tile x tile blocks from token 0 (the last block
 * of each axis ragged when tile does not divide N), writes to counts[0..2]
 * (int64, caller-owned DEVICE memory, 8-byte aligned) the number of blocks
 * whose token pairs are all live, some live, and none live. Partial blocks are
 * the ones such a kernel must mask element by element; a tile that divides the
 * frame's token span leaves none. tile: a positive multiple of 16.
 * Asynchronous on `stream`. Errors: VDIT_ERR_INVALID, VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_plan_block_census(const vdit_plan *plan, int32_t tile, int64_t *counts,
                                            void *stream);

/* Free the plan and its device buffers (synchronous w.r.t. the device). NULL is ignored. */
VDIT_API void vdit_plan_destroy(vdit_plan *plan);

/* Bytes of device workspace vdit_key_stats needs for these sizes. */
VDIT_API size_t vdit_key_stats_workspace_size(int32_t B, int32_t H, int32_t N, int32_t D);

/* Per-head key statistics and static-max eligibility ("Unchaining the Softmax"):
 *   k_mean[b,h,:]  = c   = (1/N) sum_j k_j                       fp32 [B, H, D]
 *   k_rmax[b,h]    = R   = max_j |k_j - c|_2                     fp32 [B, H]
 *   q_nmax[b,h]    = Qm  = max_i |q_i|_2                         fp32 [B, H]
 *   gap_bound[b,h] = G   = 2 * scale * Qm * R                    fp32 [B, H]
 *   eligible[b,h]  = (G <= tau) ? 1 : 0                          uint8 [B, H]
 * G bounds, for every row and every mask, how far the row's static bound can
 * sit above its true max logit; tau = 64 keeps every row's largest term above
 * e^-64, far from fp32 underflow. scale: finite and > 0; tau >= 0 (+inf makes
 * every head eligible). q, k: bf16 device tensors (see conventions).
 * workspace: device buffer of at least vdit_key_stats_workspace_size bytes,
 * caller-owned, contents need not be initialised. Reductions run in a fixed
 * order: results are bitwise reproducible. Outputs are dense, caller-owned
 * device arrays. Errors: VDIT_ERR_INVALID, VDIT_ERR_UNSUPPORTED, VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_key_stats(const void *q, const void *k, int32_t B, int32_t H, int32_t N,
                           int32_t D, const int64_t q_strides[3], const int64_t k_strides[3],
                           float scale, float tau, float *k_mean, float *k_rmax, float *q_nmax,
                           float *gap_bound, uint8_t *eligible, void *workspace,
                           size_t workspace_bytes, void *stream);

/* Allocation-free vdit_key_stats. The source pages have no counterpart to this
 * entry point; it exists for callers that may not allocate device memory at
 * all: plugins whose host framework owns every device buffer and forbids
 * cudaMalloc, or latency-critical loops that cannot afford cudaMalloc's
 * implicit device synchronisation. Same arguments, outputs and results as
 * vdit_key_stats, without the workspace: the scratch comes from a 4 MiB array
 * compiled into the library, resident on every GPU that loads it until the
 * process exits. Sizes with B*H*ceil(N/512)*(D+2)*4 > 4 MiB are rejected with
 * VDIT_ERR_INVALID before any launch. The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture. All calls share the array
 * and it keeps the last call's contents (every slot is rewritten before it is
 * read); calls whose kernels overlap on the GPU race on it and must be
 * ordered by the caller. Calls no cudaMalloc/cudaFree. */
VDIT_API vdit_status vdit_key_stats_noalloc(const void *q, const void *k, int32_t B, int32_t H,
                                            int32_t N, int32_t D, const int64_t q_strides[3],
                                            const int64_t k_strides[3], float scale, float tau,
                                            float *k_mean, float *k_rmax, float *q_nmax,
                                            float *gap_bound, uint8_t *eligible, void *stream);

/* The attention ("Deleting the Mask" + "Unchaining the Softmax"): for every
 * query token i of every head,
 *   O_i   = sum_{j in J(i)} softmax_j(scale * q_i . k_j) v_j
 *   LSE_i = ln sum_{j in J(i)} exp(scale * q_i . k_j)
 * with J(i) the plan's live keys. q, k, v: bf16 [B, H, N, D] device tensors,
 * N = the plan's num_tokens. o: [B, H, N, D], bf16 (o_dtype = VDIT_O_BF16) or
 * fp32 (VDIT_O_F32), with its own strides. lse: fp32 [B, H, N] dense, or NULL.
 * mode: VDIT_MODE_AUTO uses the static bound on heads with eligible[b,h] != 0
 * and online softmax elsewhere; FORCE_ONLINE uses online softmax everywhere
 * (k_mean, k_rmax, eligible may be NULL); FORCE_STATIC uses the bound on every
 * head (eligible may be NULL; on ineligible heads terms may underflow).
 * scale: finite and > 0. o and lse must not share memory with q, k or v (the
 * kernel reads q, k, v tiles while other CTAs write o).
 * k_mean, k_rmax: outputs of vdit_key_stats for the same k. A kernel whose
 * bounded wait expires stops early, leaving O and LSE partly unwritten, and sets
 * the plan's status word: the call itself returns before the kernel runs and
 * cannot report it, so check vdit_plan_status after the stream has passed the
 * call wherever a truncated result must not be used. The result is deterministic: two identical calls write
 * identical bytes. When the plan has gathered tiles (n_gathers > 0) the call
 * makes two launches on `stream`: the tile pairs, then the gathered tiles as a
 * programmatic dependent launch that may start while the first is still
 * running and completes only after it; work the stream orders after the call
 * follows both, and the pair can be captured in a CUDA graph.
 * Errors: VDIT_ERR_INVALID, VDIT_ERR_UNSUPPORTED, VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_attn_fwd(const vdit_plan *plan, const void *q, const void *k, const void *v,
                          void *o, int32_t o_dtype, float *lse, int32_t B, int32_t H, int32_t D,
                          const int64_t q_strides[3], const int64_t k_strides[3],
                          const int64_t v_strides[3], const int64_t o_strides[3], float scale,
                          const float *k_mean, const float *k_rmax, const uint8_t *eligible,
                          int32_t mode, void *stream);

/* ---------------------------------------------------------------------------
 * The design before frame alignment, kept as an ablation ("Deleting the Mask",
 * Fig. 3). Before the fix the pages describe, the kernel tiled the sequence in
 * multiples of 128 that ignore frame boundaries: live blocks straddled frames,
 * so the blocks that came out partial needed a mask predicate in the inner
 * loop, and the sequence was padded so that the block grid covered it; and the
 * frame window and the reference frame ran as two separate attention passes
 * writing full-precision intermediates that a merge pass re-read. These calls
 * compute the same attention as vdit_attn_fwd that way, so the cost of each
 * piece can be measured against the frame-aligned single pass.
 * ------------------------------------------------------------------------- */

/* vdit_attn_fwd with the frame-blind tiling: query blocks of 256 rows (two
 * 128-row tiles) and 128-key tiles at fixed multiples of 128 over the sequence
 * padded to a multiple of 128 (rows and keys beyond N are read as zeros and
 * never stored). Each block visits every 128-key tile holding a live key of
 * one of its rows; in a tile where some row of a warp also sees dead keys, each
 * element of S is tested against that row's live key runs and dead ones are
 * set to -inf before the softmax. Uses the plan's mask geometry and part (a
 * plan of vdit_attn_plan_part runs that part alone: rows that see no key of it
 * get O = 0 and LSE = -inf); its block schedule is not used. Arguments,
 * outputs, tolerances and errors as vdit_attn_fwd. */
VDIT_API vdit_status vdit_attn_fwd_tiles128(const vdit_plan *plan, const void *q, const void *k,
                                            const void *v, void *o, int32_t o_dtype, float *lse,
                                            int32_t B, int32_t H, int32_t D,
                                            const int64_t q_strides[3], const int64_t k_strides[3],
                                            const int64_t v_strides[3], const int64_t o_strides[3],
                                            float scale, const float *k_mean, const float *k_rmax,
                                            const uint8_t *eligible, int32_t mode, void *stream);

/* Bytes of device workspace vdit_attn_fwd_two_pass needs: fp32 O and LSE of
 * both passes, 2 * (B*H*N*D + B*H*N) * 4 bytes (each array 256-byte aligned). */
VDIT_API size_t vdit_attn_two_pass_workspace_size(int32_t B, int32_t H, int32_t N, int32_t D);

/* The attention of the whole mask in two passes and a merge: pass a runs
 * plan_window (vdit_attn_plan_part with VDIT_PART_WINDOW), pass b runs
 * plan_reference (VDIT_PART_REFERENCE of the same F, T, W, ref), each writing
 * fp32 O and LSE into the workspace; the merge kernel re-reads both and, per
 * row, with M = max(LSE_a, LSE_b) and w_x = exp(LSE_x - M), writes
 *   O = (w_a O_a + w_b O_b) / (w_a + w_b),  LSE = M + ln(w_a + w_b)
 * into o (bf16 or fp32, o_strides) and lse (fp32 [B, H, N] dense, or NULL);
 * rows whose frame sees no key of pass b take pass a unchanged. Both passes use
 * the same per-head statistics and mode. tiles = VDIT_TILES_FRAME runs both
 * passes with the frame-aligned kernel (vdit_attn_fwd), VDIT_TILES_128 with the
 * frame-blind tiling (vdit_attn_fwd_tiles128). workspace: at least
 * vdit_attn_two_pass_workspace_size bytes of caller-owned device memory,
 * 256-byte aligned. Asynchronous on `stream`. Errors: VDIT_ERR_INVALID (plans
 * that are not the two parts of one mask, workspace, arguments),
 * VDIT_ERR_UNSUPPORTED, VDIT_ERR_CUDA, and those of vdit_attn_fwd. */
VDIT_API vdit_status vdit_attn_fwd_two_pass(const vdit_plan *plan_window, const vdit_plan *plan_reference,
                                            const void *q, const void *k, const void *v, void *o,
                                            int32_t o_dtype, float *lse, int32_t B, int32_t H, int32_t D,
                                            const int64_t q_strides[3], const int64_t k_strides[3],
                                            const int64_t v_strides[3], const int64_t o_strides[3],
                                            float scale, const float *k_mean, const float *k_rmax,
                                            const uint8_t *eligible, int32_t mode, int32_t tiles,
                                            void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace vdit_key_stats_framed needs for this plan and sizes. */
VDIT_API size_t vdit_key_stats_framed_workspace_size(const vdit_plan *plan, int32_t B, int32_t H,
                                                     int32_t D);

/* Key statistics with the bound tightened per query segment ("Unchaining the
 * Softmax": the bound stays valid under windowed masks, where rows of different
 * frames attend to different subsets of the keys). For every segment s of the
 * plan (frames sharing one key-run list; one frame for sparse windows, the
 * whole sequence when dense):
 *   k_mean[b,h,:]       = c, the mean of all N keys of the head    fp32 [B, H, D]
 *   seg_rmax[b,h,s]     = max |k_j - c| over the keys s sees        fp32 [B, H, nseg]
 *   seg_gap[b,h,s]      = 2 * scale * (max |q_i| over s's rows) * seg_rmax
 *   seg_eligible[b,h,s] = seg_gap <= tau                           uint8 [B, H, nseg]
 * Never looser than vdit_key_stats (equal when a segment sees every key).
 * q, k: bf16 [B, H, N, D] device tensors, N = the plan's num_tokens. workspace:
 * at least vdit_key_stats_framed_workspace_size bytes of caller-owned device
 * memory. Fixed-order reductions (bitwise reproducible). Errors:
 * VDIT_ERR_INVALID, VDIT_ERR_UNSUPPORTED, VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_key_stats_framed(const vdit_plan *plan, const void *q, const void *k,
                                           int32_t B, int32_t H, int32_t D,
                                           const int64_t q_strides[3], const int64_t k_strides[3],
                                           float scale, float tau, float *k_mean, float *seg_rmax,
                                           float *seg_gap, uint8_t *seg_eligible, void *workspace,
                                           size_t workspace_bytes, void *stream);

/* vdit_attn_fwd with the per-segment bound and eligibility of
 * vdit_key_stats_framed (same plan) in place of the per-head ones: each work
 * unit reads R and eligibility of its own segment. Same outputs, layout,
 * determinism and errors as vdit_attn_fwd. */
VDIT_API vdit_status vdit_attn_fwd_framed(const vdit_plan *plan, const void *q, const void *k,
                                          const void *v, void *o, int32_t o_dtype, float *lse,
                                          int32_t B, int32_t H, int32_t D,
                                          const int64_t q_strides[3], const int64_t k_strides[3],
                                          const int64_t v_strides[3], const int64_t o_strides[3],
                                          float scale, const float *k_mean, const float *seg_rmax,
                                          const uint8_t *seg_eligible, int32_t mode, void *stream);

/* ---------------------------------------------------------------------------
 * Fused pre-attention chain ("Layout Is the ABI", Fig. 5). Attention's inputs
 * come out of a chain of small steps -- normalisation, projections, rotary
 * embeddings, head packing -- and the pages fuse that chain into one kernel
 * that writes its result directly in the layout the next consumer reads, so
 * no repack copies sit in between. Here the consumer is vdit_attn_fwd and the
 * layout is [B, H, N, D]. For a token row x (length C) at position n:
 *   y     = x / sqrt(mean_c x_c^2 + eps) * gamma                  (RMSNorm)
 *   z     = W y,  W = [Wq; Wk; Wv] of shape [3*H*D, C], rows head-major
 *   v_h   = z[2HD + hD + d]
 *   q_h, k_h = z[hD + d], z[HD + hD + d], each rotated pairwise:
 *           (u_i, u_{i+D/2}) -> (u_i cos a - u_{i+D/2} sin a, u_i sin a + u_{i+D/2} cos a)
 *           with a = theta[n, i], i < D/2.
 * The pages name the steps but not their variants; the readings taken are
 * RMSNorm with a learned per-channel gain on the hidden state, one fused
 * q/k/v projection without bias, and rotate-half rotary embedding of q and k
 * with a caller-supplied angle table (vdit_rope_table builds the 1-D one,
 * theta[n, i] = n * base^(-2i/D)).
 *
 * GPU mapping: the gain folds into the weights once (vdit_qkv_fold_gamma);
 * per call, a pre-pass computes 1/rms of every row and one persistent tcgen05
 * GEMM computes x W'^T with the 1/rms scale, the rotation, the bf16 rounding
 * and the head scatter in its epilogue (TMA stores into q, k, v).
 * ------------------------------------------------------------------------- */

/* w_folded[o, c] = bf16(fp32(w[o, c]) * gamma[c]), rounded to nearest-even
 * (the fp32 product is itself rounded to nearest). w, w_folded: bf16 [rows, C]
 * dense device arrays (may alias); gamma: fp32 [C] device array. Done once per
 * weight set. Errors: VDIT_ERR_INVALID (null pointer, rows < 1, C < 1),
 * VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_qkv_fold_gamma(const void *w, const float *gamma, void *w_folded,
                                         int64_t rows, int32_t C, void *stream);

/* Rotary angle table for positions n in [0, N) and pairs i in [0, D/2):
 *   table[(i * N + n) * 2 + 0] = cos(n * base^(-2i/D)),
 *   table[(i * N + n) * 2 + 1] = sin(n * base^(-2i/D)),
 * evaluated in fp64 and rounded to fp32 (layout [D/2][N][2], pair-major so
 * that consecutive rows read consecutive entries). Any other angle schedule
 * (e.g. per-axis angles for frame, height and width) may be written into the
 * same layout by the caller. Errors: VDIT_ERR_INVALID (null table, N < 1,
 * D odd or < 2, base not finite and > 0), VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_rope_table(float *table, int32_t N, int32_t D, double base, void *stream);

/* Bytes of device workspace vdit_qkv_prologue needs: one status word and one
 * fp32 per token row. */
VDIT_API size_t vdit_qkv_workspace_size(int32_t B, int32_t N);

/* The fused chain above for every row of x.
 *   x:        bf16, element (b, n, c) at x[b*x_strides[0] + n*x_strides[1] + c]
 *   w_folded: bf16 [3*H*D, C] dense, the output of vdit_qkv_fold_gamma
 *   rope:     fp32 [D/2][N][2] angle table (see vdit_rope_table)
 *   q, k, v:  bf16 [B, H, N, D] outputs, strides in elements for (b, h, n)
 *   eps:      RMSNorm epsilon (finite, >= 0)
 *   workspace: >= vdit_qkv_workspace_size(B, N) bytes of device memory; its
 *             status word must be zero at launch (it is after a fresh cudaMemset
 *             and after vdit_qkv_status).
 * Requirements: D in {64, 128}; C a multiple of 8; x strides, q/k/v strides
 * positive multiples of 8 elements; every base address 16-byte aligned.
 * Accumulation is fp32 over bf16 products; outputs are rounded once to bf16.
 * Errors: VDIT_ERR_INVALID, VDIT_ERR_UNSUPPORTED (D), VDIT_ERR_CUDA; an expired
 * wait inside the GEMM is reported by vdit_qkv_status. */
VDIT_API vdit_status vdit_qkv_prologue(const void *x, const int64_t x_strides[2],
                                       const void *w_folded, const float *rope, void *q, void *k,
                                       void *v, const int64_t q_strides[3],
                                       const int64_t k_strides[3], const int64_t v_strides[3],
                                       int32_t B, int32_t N, int32_t C, int32_t H, int32_t D,
                                       float eps, void *workspace, size_t workspace_bytes,
                                       void *stream);

/* Synchronise `stream`, then report and clear the status word in a prologue
 * workspace. *code receives the raw word (0 = none). Returns VDIT_OK when the
 * word was 0, VDIT_ERR_TIMEOUT otherwise. */
VDIT_API vdit_status vdit_qkv_status(void *workspace, void *stream, int32_t *code);

/* ---------------------------------------------------------------------------
 * Head-group pipelining over host-resident tensors ("Hiding the Collective",
 * Fig. 2). The pages split attention's heads into independent groups, each
 * with its own transfer -> attention -> transfer chain, so that every middle
 * transfer hides behind another group's attention and only the first transfer
 * in and the last transfer out stay exposed. Splitting by heads leaves the
 * token order, and so the mask, unchanged: grouped results equal ungrouped
 * ones bit for bit. Here the transfer is the host link of one GPU: a pipeline
 * copies each group's Q, K, V in, runs vdit_key_stats and vdit_attn_fwd on it,
 * and copies its O (and LSE) out, on internal streams ordered by events, with
 * two device slots in turn.
 * ------------------------------------------------------------------------- */
typedef struct vdit_pipeline vdit_pipeline;

/* The head-group schedule that vdit_pipeline_create picks for H heads when
 * groups = 0 and group_heads is NULL: writes the head count of each group to
 * out[0 .. n-1] (host array of cap entries) and returns n, or returns 0 and
 * writes nothing when H < 1, out is NULL or cap < n. Host only: no device
 * work, no allocation, callable without a GPU. */
VDIT_API int32_t vdit_pipeline_default_groups(int32_t H, int32_t *out, int32_t cap);

/* Create a pipeline for attention with `plan` over B x H heads of size D, split
 * into `groups` head groups: group_heads[g] heads each (host array of `groups`
 * positive counts summing to H), or, when group_heads is NULL, ceil(H / groups)
 * heads each (the last may be smaller). groups = 0 with group_heads NULL picks
 * a tapered schedule: 1, 2, 3 heads, then groups of 4 (the heads left over
 * spread one at a time over those groups, so a middle group holds up to 7 heads
 * when there are fewer middle groups than leftover heads, e.g. 1,2,3,7,3,2,1 for
 * H = 19), then 3, 2, 1 heads, so that the exposed first copy-in and last
 * copy-out are one head each; for H < 16, and for H >= 248 (where the tapered
 * schedule would need more than 64 groups), an even split into groups of about 4. Allocates two device slots (Q, K, V, O,
 * LSE, statistics and their workspace for the largest group each), four streams
 * and the events; owns them until vdit_pipeline_destroy. Errors:
 * VDIT_ERR_INVALID (null plan or out, B or H < 1, groups outside [0, H], bad
 * group_heads, plan from another device), VDIT_ERR_UNSUPPORTED (D),
 * VDIT_ERR_NOMEM, VDIT_ERR_CUDA. */
VDIT_API vdit_status vdit_pipeline_create(const vdit_plan *plan, int32_t B, int32_t H, int32_t D,
                                          int32_t groups, const int32_t *group_heads,
                                          vdit_pipeline **out);

/* Run attention on HOST tensors: q_host, k_host, v_host (bf16, read) and o_host
 * (bf16, written) share the element strides host_strides for (b, h, n), with d
 * contiguous; lse_host (fp32 [B, H, N] dense) may be NULL. Host memory should be
 * pinned (page-locked) for the copies to overlap the kernels. Key statistics
 * use tau as in vdit_key_stats; mode as in vdit_attn_fwd. Asynchronous with
 * respect to the host: the work is ordered after everything already queued on
 * `stream`, and `stream` waits for all of it, so a synchronisation of `stream`
 * means o_host (and lse_host) are complete; every host buffer stays owned by
 * the caller and must stay valid until then. An expired wait inside attention
 * is reported only by vdit_plan_status on the plan: this call cannot see it (the
 * kernels run after it returns), so a caller that must not use a truncated O
 * calls vdit_plan_status after the stream has passed the run. Arguments
 * (pointers, strides, scale finite and > 0, tau >= 0, mode) are checked before
 * anything is queued.
 * Consecutive batches overlap when they run on two pipelines, each with its
 * own plan, on two streams: one batch's first copy-in and last copy-out then
 * run beside the other batch's kernels (+6% at the 720p-like shape).
 * An error from a later step returns at once; copies and kernels of earlier
 * groups may still be in flight, and `stream` is made to wait for all of them,
 * so the host buffers must stay valid until `stream` is synchronised, as on
 * success. A pipeline may be driven from different streams in turn: a run
 * reuses a device slot only after the previous run's kernels and copies of that
 * slot are done. Errors: VDIT_ERR_INVALID,
 * VDIT_ERR_CUDA, and those of vdit_key_stats and vdit_attn_fwd. */
VDIT_API vdit_status vdit_pipeline_run(vdit_pipeline *pipeline, const void *q_host,
                                       const void *k_host, const void *v_host, void *o_host,
                                       float *lse_host, const int64_t host_strides[3], float scale,
                                       float tau, int32_t mode, void *stream);

/* Wait for the pipeline's streams, then free its device memory, streams and
 * events. NULL is ignored. */
VDIT_API void vdit_pipeline_destroy(vdit_pipeline *pipeline);

/* Failure-detection test hook. Every wait inside the attention kernel and the
 * prologue GEMM is bounded; when a wait expires the kernel records which wait
 * in its status word (the plan's, or the prologue workspace's), drains its
 * in-flight copies and MMAs, frees its tensor memory and exits early
 * (vdit_plan_status / vdit_qkv_status then return VDIT_ERR_TIMEOUT). This sets
 * the bound for kernels launched afterwards, process-wide: ns = 0 restores the
 * default of one second. A tiny bound makes a normal call expire on purpose,
 * so the early-exit path can be tested without any fault. Draining always
 * keeps the default bound. */
VDIT_API void vdit_set_wait_limit_ns(uint64_t ns);

/* Allocation-failure test hook. With n >= 1, the n-th device allocation the
 * library makes from now on (counted process-wide; plan and pipeline creation
 * allocate) fails as if the device were out of memory, once; the call that
 * made it frees what it had allocated and returns VDIT_ERR_NOMEM. n <= 0
 * switches the hook off. For tests of the error paths; no fault is involved. */
VDIT_API void vdit_set_alloc_fail_after(int32_t n);

/* Launch-failure test hook. With n >= 1, the n-th attention launch from now on
 * (vdit_attn_fwd, vdit_attn_fwd_framed, and those inside vdit_pipeline_run;
 * counted process-wide) is refused before anything is launched, once, as if
 * the launch had failed: the call returns VDIT_ERR_CUDA. n <= 0 switches the
 * hook off. For tests of the error paths (e.g. a pipeline run that fails part-
 * way); no fault is involved. */
VDIT_API void vdit_set_launch_fail_after(int32_t n);

/* Thread-local, library-owned text of the last error on this thread ("" if none). */
VDIT_API const char *vdit_last_error(void);

/* Library version string. */
VDIT_API const char *vdit_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VDIT_H */

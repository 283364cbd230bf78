// Host-side internals shared by the libvdit translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <string>

#include "vdit.h"

namespace vdit {

// Thread-local error text behind vdit_last_error().
void set_error(const char *fmt, ...);
void clear_error();

// Formats a CUDA error into the thread-local message and returns VDIT_ERR_CUDA.
vdit_status cuda_fail(cudaError_t e, const char *what);

#define VDIT_CUDA_TRY(expr)                                      \
    do {                                                         \
        cudaError_t e__ = (expr);                                \
        if (e__ != cudaSuccess) return ::vdit::cuda_fail(e__, #expr); \
    } while (0)

// Bound on every spin-wait inside a kernel, set by vdit_set_wait_limit_ns
// (default one second); draining after an expired wait always uses the default.
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;
unsigned long long wait_limit_ns();

// cudaMalloc behind the allocation-failure test hook (vdit_set_alloc_fail_after):
// every device allocation the library makes goes through here.
cudaError_t device_alloc(void **ptr, size_t bytes);

// Launch-failure test hook (vdit_set_launch_fail_after): true for the one
// attention launch that is to fail as if the launch had been refused.
bool launch_fails_by_hook();

// Query-tile geometry shared by the plan and the attention kernel.
constexpr int kTileRows = 128;   // rows of one query tile (tcgen05 M)
constexpr int kTilesPerUnit = 2; // query tiles that share one K/V stream
constexpr int kSegInts = 8;      // ints per segment record
constexpr int kMaxFrames = 4096; // frames a plan may hold
constexpr int kMaxClasses = 64;  // distinct unit costs a plan may hold
constexpr int kMaxPairsPerSegment = 1 << 16;  // tile pairs a segment may hold (16-bit field)
// Gathered tiles: the ragged last rows of several segments (each a multiple of
// 16 rows, at most kGatherMaxRows, of a segment of at least kGatherMinSegRows
// rows) share one 128-row query tile. A record holds its piece count, rows, the
// union of the pieces' key runs and the pieces.
constexpr int kGatherMaxPieces = 8;
constexpr int kGatherMaxRows = 64;
constexpr int kGatherMinSegRows = 8 * kTileRows;
// Tail tiles: a plan without gathered tiles, with at least kTailMinPairs tile
// pairs per head, runs the tiles of its last kTailPairs pairs as one-piece
// records in the same second launch.
constexpr int kTailPairs = 8;
constexpr int kTailMinPairs = 32;
constexpr int kGatherPiece = 8;                                  // first piece: seg, row0, rows
constexpr int kGatherInts = kGatherPiece + 3 * kGatherMaxPieces; // ints per gathered-tile record

// A scale factor the kernels can use: positive and finite (NaN and +inf fail).
inline bool finite_positive(float x) { return x > 0.f && x <= 3.402823466e38f; }

// Header the schedule kernel writes (device), read back once by the host.
struct PlanHeader {
    long long nnz;
    long long live_pairs;
    int n_segments;
    int n_units;
    int n_classes;
    int error; // non-zero: the kernel found an inconsistent request
    int n_gathers;
};

}  // namespace vdit

struct vdit_plan {
    int F, T, W, ref, bs, dense;
    int part = VDIT_PART_ALL;   // which part of the mask the plan schedules
    long long N;
    int n_qblocks;
    vdit::PlanHeader h;  // host copy of the header
    int device;
    // device buffers (owned)
    vdit::PlanHeader *d_header = nullptr;
    int32_t *d_row_ptr = nullptr;
    int32_t *d_col_idx = nullptr;
    int32_t *d_frame_runs = nullptr;
    int32_t *d_segments = nullptr;
    int32_t *d_units = nullptr;
    int32_t *d_class_off = nullptr;
    int32_t *d_gathers = nullptr;
    int32_t *d_status = nullptr;
    int units_cap = 0;
};

namespace vdit {
// Launches the two schedule kernels for `p` on `stream` (buffers must exist;
// col_idx may be null when only the meta kernel should run).
cudaError_t launch_plan_kernels(const vdit_plan *p, cudaStream_t stream, bool csr);
}  // namespace vdit

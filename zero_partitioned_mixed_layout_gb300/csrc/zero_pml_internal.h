// Internal definitions shared by the host part (host.cpp) and the CUDA part
// (zero_pml.cu) of the library: workspace layout, the per-step scalar block
// and the thread-local CUDA error record.
#pragma once

#include <cstddef>
#include <cstdint>

#include "zero_pml.h"

namespace zpml {

// 16 bytes holding a double2 (the CUDA vector type is not visible to the
// host-only translation units that include this header)
struct alignas(16) double2_storage {
    double x, y;
};

// Threads per block of every streaming kernel.
constexpr int kThreads = 256;
// Upper bound on the grid of the norm pass (one binary64 partial per block).
constexpr int kMaxBlocks = 4096;
// Elements per work item when the arrays come as a list (multiple of 8, so
// every chunk but a tensor's last starts and ends on a 16-byte boundary).
constexpr int64_t kChunk = 1 << 13;  // elements of a pass-1 list work item (one warp each)
// Elements per work item of pass 2 over a list: one block of kThreads
// threads, one 8-element vector each.
constexpr int kTileVectors = 2;  // 8-element vectors per thread of a pass-2 list tile
constexpr int64_t kTile = (int64_t)kThreads * 8 * kTileVectors;

// The scalars of one step's element update, written by the decision kernel
// and read by every block of pass 2 (binary32, as the update runs).
struct StepScalars {
    float inv_scale;  // 1 / S
    float clip;       // 1, or max_norm / (norm + 1e-6) when below 1
    float b1, omb1;   // beta1, 1 - beta1
    float b2, omb2;   // beta2, 1 - beta2
    float eps;
    float step_size;  // lr / (1 - beta1^t)
    float isb2;       // 1 / sqrt(1 - beta2^t)
    float lrwd;       // lr * weight_decay
    int32_t skip;
    int32_t pad;
    // for the bias-correction window of the next steps (see PowCache)
    double lr, beta1, beta2;
    int64_t next_t;   // step count of the next applied step
};

// The binary64 bias-correction terms of a window of kPowWindow consecutive
// step counts [t0, t0 + kPowWindow), computed ahead of time by one warp of
// pass 2 (one warp-wide pow: a lane per term) whenever the next step count
// leaves the window, and used by the decision when its tags match.  A
// binary64 pow is slow on this GPU (about 4 us for one call), so one call
// per kPowWindow steps keeps it off every step's critical path.
constexpr int kPowWindow = 16;
struct PowCache {
    int64_t t0;                   // tag: first step count of the window; 0 = empty
    double beta1, beta2;          // tags
    double lr;                    // tag of step_size
    double bc1[kPowWindow];       // 1 - beta1^t
    float step_size[kPowWindow];  // lr / bc1, rounded once
    float isb2[kPowWindow];       // 1 / sqrt(1 - beta2^t), rounded once
};

// One array set of a list: the gradient, the fp32 master / momentum /
// variance and the low-precision copy of one tensor (or one shard).
struct TensorEntry {
    const void *g;
    float *p;
    float *m;
    float *v;
    void *plp;
    int64_t numel;
};


// One work item of a list: elements [index * size, min(numel, (index+1) *
// size)) of tensor `tensor`, size being kChunk (pass 1) or kTile (pass 2).
struct WorkItem {
    int32_t tensor;
    int32_t index;
};

// Workspace layout (all offsets 128-byte aligned):
//   [0, 256)            header: reduction ticket, count of waits that gave up
//   [256, 384)          StepScalars of the current step
//   [384, 768)          PowCache: the bias corrections of a window of steps
//   [768, 768 + 16*kMaxBlocks)  per-block partials of the norm pass (double2)
//   then                GroupArea: tickets and partials of the block groups
//                       of a one-shot reduction
//   then                a list's table: TensorEntry[n], then the work
//                       items of pass 2 (one per kTile elements of each
//                       tensor) and of pass 1 (one per kChunk); a flat
//                       one-shot reduction keeps its per-block partials
//                       here instead
struct WsHeader {
    unsigned int ticket;
    // waits of a kernel that gave up (a bulk copy not landed within its
    // limit), since the workspace was zero-filled; sticky
    unsigned int stalls;
};
constexpr size_t kWsScalars = 256;
constexpr size_t kWsPowCache = 384;
constexpr size_t kWsPartials = 768;
static_assert(sizeof(StepScalars) <= kWsPowCache - kWsScalars, "StepScalars must fit its workspace slot");
static_assert(sizeof(PowCache) <= kWsPartials - kWsPowCache, "PowCache must fit its workspace slot");

// A one-shot reduction's blocks report in groups of kGroupBlocks: the last
// block of a group sums the group's partials in block order, the last group
// to finish sums the group partials in group order.  Its tickets start at
// zero (a fresh workspace is zero-filled) and every finisher resets its own.
constexpr int kGroupBlocks = 1024;
constexpr int kMaxGroups = 4096;
struct GroupArea {
    unsigned int tickets[kMaxGroups];
    double2_storage partials[kMaxGroups];
};
constexpr size_t kWsGroups = kWsPartials + 16 * (size_t)kMaxBlocks;
constexpr size_t kWsTable = (kWsGroups + sizeof(GroupArea) + 255) & ~(size_t)255;

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Bytes of the table region: a list's table for up to n_tensors tensors of
// total_numel elements (entries, pass-2 tiles, pass-1 chunks; each tensor
// adds at most one partial item to each), and at least one 16-byte partial
// per 4096 elements of a flat pass over total_numel elements.
inline size_t table_bytes(int64_t n_tensors, int64_t total_numel)
{
    const size_t list = align256((size_t)n_tensors * sizeof(TensorEntry)) +
                        align256((size_t)(total_numel / kTile + n_tensors + 1) * sizeof(WorkItem)) +
                        align256((size_t)(total_numel / kChunk + n_tensors + 1) * sizeof(WorkItem));
    const size_t flat = align256((size_t)(total_numel / 256) + 256);
    return list > flat ? list : flat;
}

// Records a CUDA error message for zero_strerror on this thread.
void set_cuda_error(const char *what, int cuda_code, const char *cuda_msg);

}  // namespace zpml

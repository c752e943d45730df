// Internal definitions shared by the host plan code and the CUDA kernels of
// libtide.  Not part of the C ABI (see include/tide.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/tide.h"

namespace tide {

// NVTX range for the lifetime of a scope (header-only NVTX v3: a no-op unless
// a profiler is attached), so that profilers can select the library's calls.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr int kMaxWorld = 1024;
constexpr int kFoldThreads = 256;            // threads per fold CTA (direct kernel)
constexpr int kBulkConsumerWarps = 4;        // bulk kernel: warp 0 produces, warps 1..4 consume
constexpr int kBulkThreads = 32 * (1 + kBulkConsumerWarps);
// A bulk CTA that has an SM to itself (small CTA budgets) runs 8 consumer
// warps with 4 vectors each and copies 16 KB per rank (every order but the
// tree order, whose per-level partials take the registers).
constexpr int kBulkConsumerWarpsWide = 8;
#ifndef TIDE_BULK_RING_KB
#define TIDE_BULK_RING_KB 96
#endif
constexpr int kBulkSmemTarget = TIDE_BULK_RING_KB * 1024;  // stage ring bytes per bulk CTA (96 KB: two CTAs per SM)
constexpr uint64_t kWaitBudgetNs = 4000000000ull;   // bounded mbarrier waits: 4 s
constexpr uint64_t kShortWaitBudgetNs = 50000000ull; // with TIDE_DEBUG_SHORT_WAIT: 50 ms
constexpr int kAgThreads = 256;              // threads per placement CTA
constexpr int kAgParamsPerLaunch = 1024;     // full[] pointers passed by value per placement launch
constexpr int64_t kDefaultChunkBytes = 16384;  // bf16 bytes per rank per fold work item
constexpr int64_t kAgChunkElems = 16384;     // bf16 elements per placement work item

// One (parameter, rank) shard piece.  Element offsets; the output address is
// out_base + rank * stride + dst_elem, the source address of rank u is
// ptrs[param * W + u] + src_elem.
struct Seg {
    int64_t src_elem;
    int64_t dst_elem;
    int64_t n_valid;
    int64_t n_pad;
    int32_t param;
    int32_t rank;
    int32_t src_phase;  // (address / element size) mod (16 / element size) of every rank's first element, -1 if ranks differ
    int32_t pad_;
};
static_assert(sizeof(Seg) == 48, "Seg layout");

// One work item: `count` elements starting `begin` elements into the piece's
// real data (kind 0) or into its padding (kind 1).
struct Item {
    int32_t seg;
    uint32_t count_kind;  // bit 31: padding item; bits 0..30: count
    int64_t begin;
};
static_assert(sizeof(Item) == 16, "Item layout");
constexpr uint32_t kItemPad = 0x80000000u;

struct FoldParams {
    const uint64_t *ptrs;  // [P * W] gradient base pointers
    const Seg *segs;
    const Item *items;
    int64_t n_items;
    float *out;
    int64_t stride;
    float alpha;
    int32_t world;
    int32_t sched;
    uint32_t *counters;    // [2] dynamic-schedule ticket and done counters
    int32_t *status;       // device status word
    uint32_t debug;
    // bulk kernel only
    uint64_t wait_budget_ns;  // bound on every mbarrier wait
    int32_t fill_elems;       // elements per rank per stage fill (multiple of 8)
    int32_t fill_ranks;       // ranks per stage fill
    int32_t stages;           // ring depth
    int32_t order;            // TIDE_ORDER_*
    int32_t node_size;        // ranks per node of TIDE_ORDER_NODES
    int32_t dtype;            // TIDE_DTYPE_* of the gradients
    int32_t consumer_warps;   // kBulkConsumerWarps or kBulkConsumerWarpsWide (bulk_consumer_warps)
};

// Stage geometry of the bulk kernel for a world size.
struct BulkShape {
    int32_t fill_elems;
    int32_t fill_ranks;
    int32_t stages;
    size_t smem_bytes;
};
// fill_elems / fill_ranks 0 = default; whole_sm: the grid has at most one CTA per SM
BulkShape bulk_shape(int world, int64_t fill_elems, int fill_ranks, bool whole_sm, int elem_bytes,
                     int order = TIDE_ORDER_RANK_ASC);
// Tree order: partials of complete stage fills are kept per level of a
// binary counter in registers, so a chunk holds at most 2^kTreeLevels - 1
// full fills.
constexpr int kTreeLevels = 8;

// Placement kernel parameters, passed by value: NP destination pointers.
// Launches for at most kAgParamsSmall parameters use the small form (a
// 0.4 KB parameter block instead of 8 KB, which shortens every launch).
template <int NP>
struct AgParamsT {
    const Seg *segs;
    const Item *items;
    int64_t item_begin, item_end;  // this launch's item range
    const uint16_t *slots;
    const float *slots_f32;        // mixed-precision placement: fp32 slots (slots unused)
    int64_t stride;
    int32_t param_base;            // full[0] is parameter param_base
    int32_t n_full;
    uint16_t *full[NP];
};
using AgParams = AgParamsT<kAgParamsPerLaunch>;
constexpr int kAgParamsSmall = 32;

// Launchers (rs_fold.cu / ag_place.cu).  Return cudaGetLastError() of the launch.
cudaError_t launch_fold(const FoldParams &fp, int kernel, int accumulate, int grid, int block, size_t smem,
                        cudaStream_t stream);
cudaError_t fold_occupancy(int kernel, int world, int block, size_t smem, int *blocks_per_sm,
                           int dtype = TIDE_DTYPE_BF16, int order = TIDE_ORDER_RANK_ASC, int fill_ranks = 0,
                           int consumer_warps = kBulkConsumerWarps);
// Consumer warps of the bulk kernel for a launch shape.
inline int bulk_consumer_warps(bool whole_sm, int order, int dtype)
{
    (void)dtype;
    return whole_sm && order != TIDE_ORDER_TREE ? kBulkConsumerWarpsWide : kBulkConsumerWarps;
}
size_t fold_smem_bytes(int kernel, int world, int64_t fill_elems, int fill_ranks, bool whole_sm,
                       int elem_bytes = 2, int order = TIDE_ORDER_RANK_ASC);
cudaError_t launch_ag(const AgParams &ap, int grid, cudaStream_t stream);
cudaError_t launch_ag_f32(const AgParams &ap, int grid, cudaStream_t stream);

extern std::atomic<uint64_t> g_launches;

// Device address of the allocation-free fold's status word on device `dev`
// (rs_fold_noalloc.cu), or NULL before that entry point's first call there.
int32_t *noalloc_status_word(int dev);

// Set the detail message tide_last_error() returns on this thread.  The
// message is copied into a fixed per-thread buffer, so callers may rely on
// it not allocating once the thread's buffer exists.
void record_error(const char *msg);

}  // namespace tide

struct tide_plan {
    int32_t world = 0;
    int32_t nparams = 0;
    int64_t slot_numel = 0;
    std::vector<int64_t> dim0, row_numel, rows, offset;
    std::vector<uint64_t> ptrs;          // [P * W]
    std::vector<tide::Seg> segs;         // [P * W], param-major
    std::vector<tide::Item> rs_items;
    std::vector<tide::Item> ag_items;    // real data only, ordered by parameter
    std::vector<int64_t> ag_param_item_begin;  // [P + 1]
    tide_plan_flags_t flags{};
    int64_t chunk_elems = 0;
    int32_t grid = 0, block = 0, sms = 0;
    size_t fold_smem = 0;
    int kernel = TIDE_KERNEL_DIRECT;
    int elem_bytes = 2;                  // gradient element size (bf16 2, fp32 4)
    bool whole_sm = false;               // bulk kernel: at most one CTA per SM (deeper ring)
    int consumer_warps = tide::kBulkConsumerWarps;  // bulk kernel: consumer warps per CTA
    bool host_only = false;
    bool host_grads = false;             // some gradients are page-locked host memory (direct kernel only)
    std::vector<uint8_t> ptr_host;       // [P * W]: that gradient is page-locked host memory
    int device = -1;
    uintptr_t src_lo = 0, src_hi = 0;    // hull of all gradient ranges
    // device side
    void *d_block = nullptr;
    uint64_t *d_ptrs = nullptr;
    tide::Seg *d_segs = nullptr;
    tide::Item *d_rs_items = nullptr;
    tide::Item *d_ag_items = nullptr;
    uint32_t *d_counters = nullptr;
    int32_t *d_status = nullptr;
    cudaEvent_t last_use = nullptr;
    // copy-engine placement: internal streams, fork / join events
    int32_t n_ce = 0;
    cudaStream_t ce_stream[8] = {};
    cudaEvent_t ce_fork = nullptr;
    cudaEvent_t ce_join[8] = {};
    bool captured = false;               // a launch of this plan was captured into a CUDA graph
};

// tide_rs_fold_noalloc: the reduce-scatter fold for callers that cannot
// allocate GPU memory.
//
// tide_rs_fold needs a plan, and building a plan calls cudaMalloc for the
// plan's device tables (gradient pointers, shard pieces, work items).  Some
// callers cannot do that: code that runs while a caching allocator holds its
// lock or is itself servicing an allocation (an allocator hook or an
// out-of-memory handler), code under a memory cap or custom pool that
// forbids new device allocations, and short-lived tools that must not leave
// allocations behind.  This entry point takes the parameter descriptors
// directly and keeps the tables of the call in one fixed array in device
// memory that the library owns for its whole lifetime, so a call allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// The price is a fixed size limit and shared state:
//   * the tables of one call must fit in TIDE_NOALLOC_SCRATCH_BYTES (4 MiB);
//     larger requests are rejected with TIDE_ERR_INVALID_ARG;
//   * every GPU that loads this library keeps that 4 MiB until the process
//     exits;
//   * all calls share the array, which keeps the last call's tables: calls
//     that overlap on the GPU (for example on two streams without ordering
//     between them) race and may read each other's tables.  Calls on one
//     stream are ordered and safe.
// The first call on each device (an empty one, with no parameters, will do)
// looks up the array's device address (cudaGetSymbolAddress) with that
// device current and loads the fold kernels; make that first call before any
// stream capture, outside the context that cannot allocate.
//
// The first 256 bytes of the array hold the status word of the bounded
// device-side waits (offset 0) and the dynamic schedule's two counters
// (offsets 8 and 12, zero at load; every fold resets them as it finishes);
// the tables follow.  Uploads never touch this slot: an expired wait stays
// recorded until tide_last_device_status(NULL, stream) reads and clears it
// on the current device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "tide_internal.h"

namespace {

constexpr size_t kScratchBytes = TIDE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The call's tables on every device that loads the library.  Host code must
// not pass this name to a kernel: on the host it is only a stand-in for the
// device symbol.  Its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host copy of the same tables, built in place so the call needs no heap.
alignas(256) unsigned char g_host_tables[kScratchBytes];
void *g_scratch_dev[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_lock;
constexpr size_t kStatusBytes = 256;  // status word and schedule counters at the start of the array
constexpr size_t kCountersAt = 8;     // byte offset of the two schedule counters in that slot

// Record the detail that tide_last_error() reports, without heap use.
tide_status_t noalloc_fail(tide_status_t st, const char *fmt, ...)
{
    char buf[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    tide::record_error(buf);
    return st;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Once per device, with it current (caller holds g_lock): the array's device
// address, the SM count, and the fold kernels' shared-memory attribute (which
// loads both of them), so that later calls load and look up nothing.
tide_status_t noalloc_setup(int dev)
{
    if (g_scratch_dev[dev])
        return TIDE_OK;
    void *addr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess || !addr)
        return noalloc_fail(TIDE_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) {
        const tide::BulkShape bs = tide::bulk_shape(8, 0, 0, false, 2);
        e = tide::fold_occupancy(TIDE_KERNEL_BULK, 8, tide::kBulkThreads, bs.smem_bytes, &per_sm);
    }
    if (e != cudaSuccess)
        return noalloc_fail(TIDE_ERR_CUDA, "set-up: %s", cudaGetErrorString(e));
    g_sms[dev] = sms;
    g_scratch_dev[dev] = addr;
    return TIDE_OK;
}

}  // namespace

namespace tide {
// Device address of the allocation-free fold's status word on device `dev`,
// or NULL if that entry point has not been set up on it.
int32_t *noalloc_status_word(int dev)
{
    std::lock_guard<std::mutex> guard(g_lock);
    if (dev < 0 || dev >= kMaxDevices)
        return nullptr;
    return static_cast<int32_t *>(g_scratch_dev[dev]);
}
}  // namespace tide

extern "C" tide_status_t tide_rs_fold_noalloc(int32_t world, int32_t num_params, const tide_param_desc_t *params,
                                              float *out_base, int64_t out_slot_stride, float alpha,
                                              int32_t accumulate, void *stream_)
{
    tide::record_error("");
    if (world < 1 || world > tide::kMaxWorld)
        return noalloc_fail(TIDE_ERR_INVALID_ARG, "world %d outside [1, %d]", world, tide::kMaxWorld);
    if (num_params < 0 || (num_params > 0 && !params))
        return noalloc_fail(TIDE_ERR_INVALID_ARG, "bad num_params / params");
    if (accumulate != 0 && accumulate != 1)
        return noalloc_fail(TIDE_ERR_INVALID_ARG, "accumulate must be 0 or 1");
    const int64_t CH = tide::kDefaultChunkBytes / 2;
    constexpr int64_t kLimit = int64_t(1) << 60;

    // Pass 1: geometry (dim-0 shards of R = ceil(D / W) rows, prefix offsets)
    // and the table sizes, without writing anything.
    int64_t S = 0, running = 0, n_items = 0;
    for (int32_t p = 0; p < num_params; ++p) {
        const int64_t D = params[p].dim0, K = params[p].row_numel;
        if (D < 0 || K < 0 || (K && D > kLimit / K))
            return noalloc_fail(TIDE_ERR_INVALID_ARG, "params[%d]: bad dims", p);
        const int64_t R = (D + world - 1) / world;
        if (K && R > kLimit / K / world)
            return noalloc_fail(TIDE_ERR_INVALID_ARG, "params[%d]: size overflows", p);
        const int64_t o = params[p].shard_offset == -1 ? running : params[p].shard_offset;
        // Explicit offsets must increase with p so that non-overlap is an
        // O(P) check needing no sort buffer.
        if (o < running || o > kLimit - R * K)
            return noalloc_fail(TIDE_ERR_INVALID_ARG,
                                "params[%d]: shard_offset must be -1 or at least the previous shard's end", p);
        running = o + R * K;
        S = std::max(S, running);
        for (int32_t r = 0; r < world; ++r) {
            const int64_t v = std::min(std::max(D - int64_t(r) * R, int64_t(0)), R);
            n_items += (v * K + CH - 1) / CH + ((R - v) * K + CH - 1) / CH;
        }
    }
    const size_t n_pieces = size_t(num_params) * size_t(world);
    const size_t o_ptrs = kStatusBytes;
    const size_t o_segs = o_ptrs + round256(n_pieces * sizeof(uint64_t));
    const size_t o_items = o_segs + round256(n_pieces * sizeof(tide::Seg));
    const size_t total = o_items + round256(size_t(n_items) * sizeof(tide::Item));
    if (total > kScratchBytes)
        return noalloc_fail(TIDE_ERR_INVALID_ARG,
                            "the call needs %zu bytes of tables; the allocation-free entry point holds %zu "
                            "(use tide_plan_build / tide_rs_fold instead)",
                            total, kScratchBytes);
    if (out_slot_stride < S)
        return noalloc_fail(TIDE_ERR_INVALID_ARG, "out_slot_stride %lld < S %lld", (long long)out_slot_stride,
                            (long long)S);

    std::lock_guard<std::mutex> guard(g_lock);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return noalloc_fail(TIDE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return noalloc_fail(TIDE_ERR_UNSUPPORTED, "device %d beyond %d", dev, kMaxDevices);
    const tide_status_t st = noalloc_setup(dev);  // before the early return: an empty call sets up the device
    if (st != TIDE_OK)
        return st;
    if (n_items == 0)
        return TIDE_OK;
    if (!out_base)
        return noalloc_fail(TIDE_ERR_INVALID_ARG, "out_base is NULL");
    if (reinterpret_cast<uintptr_t>(out_base) & 3u)
        return noalloc_fail(TIDE_ERR_ALIGNMENT, "out_base is not 4-byte aligned");
    if (out_slot_stride > kLimit / world)
        return noalloc_fail(TIDE_ERR_INVALID_ARG, "output extent overflows");
    const uintptr_t out_lo = reinterpret_cast<uintptr_t>(out_base);
    const uintptr_t out_hi = out_lo + uintptr_t((world - 1) * out_slot_stride + S) * 4u;

    unsigned char *scratch = static_cast<unsigned char *>(g_scratch_dev[dev]);

    // Pass 2: fill the host tables (pointers, pieces, work items).
    auto *ptrs = reinterpret_cast<uint64_t *>(g_host_tables + o_ptrs);
    auto *segs = reinterpret_cast<tide::Seg *>(g_host_tables + o_segs);
    auto *items = reinterpret_cast<tide::Item *>(g_host_tables + o_items);
    running = 0;
    int64_t it = 0;
    for (int32_t p = 0; p < num_params; ++p) {
        const int64_t D = params[p].dim0, K = params[p].row_numel, R = (D + world - 1) / world;
        const int64_t o = params[p].shard_offset == -1 ? running : params[p].shard_offset;
        running = o + R * K;
        if (!params[p].rank_base)
            return noalloc_fail(TIDE_ERR_INVALID_ARG, "params[%d].rank_base is NULL", p);
        for (int32_t u = 0; u < world; ++u) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(params[p].rank_base[u]);
            if (D * K > 0 && a == 0)
                return noalloc_fail(TIDE_ERR_INVALID_ARG, "params[%d].rank_base[%d] is NULL", p, u);
            if (a & 1u)
                return noalloc_fail(TIDE_ERR_ALIGNMENT, "params[%d].rank_base[%d] is not 2-byte aligned", p, u);
            if (D * K > 0 && out_lo < a + uintptr_t(D * K) * 2u && a < out_hi)
                return noalloc_fail(TIDE_ERR_INVALID_ARG, "the output overlaps gradient [%d][%d]", u, p);
            ptrs[size_t(p) * world + u] = a;
        }
        for (int32_t r = 0; r < world; ++r) {
            const int64_t v = std::min(std::max(D - int64_t(r) * R, int64_t(0)), R);
            tide::Seg &s = segs[size_t(p) * world + r];
            s.src_elem = int64_t(r) * R * K;
            s.dst_elem = o;
            s.n_valid = v * K;
            s.n_pad = (R - v) * K;
            s.param = p;
            s.rank = r;
            s.pad_ = 0;
            int32_t ph = -1;
            for (int32_t u = 0; u < world; ++u) {
                const int32_t x = int32_t(((ptrs[size_t(p) * world + u] >> 1) + uint64_t(s.src_elem)) & 7u);
                if (u == 0)
                    ph = x;
                else if (x != ph) {
                    ph = -1;
                    break;
                }
            }
            s.src_phase = ph;
            const int32_t si = int32_t(size_t(p) * world + r);
            for (int64_t b = 0; b < s.n_valid; b += CH)
                items[it++] = {si, uint32_t(std::min(CH, s.n_valid - b)), b};
            for (int64_t b = 0; b < s.n_pad; b += CH)
                items[it++] = {si, uint32_t(std::min(CH, s.n_pad - b)) | tide::kItemPad, b};
        }
    }

    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    // From pageable host memory: the call returns once the bytes have left
    // g_host_tables, so the next call may rewrite it.
    // The status word's slot (the first kStatusBytes) is not part of the upload.
    e = cudaMemcpyAsync(scratch + o_ptrs, g_host_tables + o_ptrs, total - o_ptrs, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return noalloc_fail(TIDE_ERR_CUDA, "table upload: %s", cudaGetErrorString(e));

    tide::FoldParams fp{};
    fp.ptrs = reinterpret_cast<const uint64_t *>(scratch + o_ptrs);
    fp.segs = reinterpret_cast<const tide::Seg *>(scratch + o_segs);
    fp.items = reinterpret_cast<const tide::Item *>(scratch + o_items);
    fp.n_items = n_items;
    fp.out = out_base;
    fp.stride = out_slot_stride;
    fp.alpha = alpha;
    fp.world = world;
    fp.sched = TIDE_SCHED_DYNAMIC;  // the default schedule, resolved below as tide_plan_build does
    fp.counters = reinterpret_cast<uint32_t *>(scratch + kCountersAt);
    fp.status = reinterpret_cast<int32_t *>(scratch);
    fp.wait_budget_ns = tide::kWaitBudgetNs;
    fp.order = TIDE_ORDER_RANK_ASC;
    fp.node_size = 0;
    fp.dtype = TIDE_DTYPE_BF16;
    // The default bulk-copy fold, as tide_plan_build would configure it.
    const tide::BulkShape bs = tide::bulk_shape(world, 0, 0, false, 2);
    fp.fill_elems = bs.fill_elems;
    fp.fill_ranks = bs.fill_ranks;
    fp.stages = bs.stages;
    fp.consumer_warps = tide::kBulkConsumerWarps;
    int per_sm = 0;
    const int sms = g_sms[dev];
    e = tide::fold_occupancy(TIDE_KERNEL_BULK, world, tide::kBulkThreads, bs.smem_bytes, &per_sm);
    if (e != cudaSuccess)
        return noalloc_fail(TIDE_ERR_CUDA, "launch geometry: %s", cudaGetErrorString(e));
    const int64_t wave = int64_t(std::max(per_sm, 1)) * sms;
    if (n_items <= wave)
        fp.sched = TIDE_SCHED_STATIC;  // every CTA gets at most one work item: no claims needed
    const int grid = int(std::min<int64_t>(wave, n_items));
    e = tide::launch_fold(fp, TIDE_KERNEL_BULK, accumulate, grid, tide::kBulkThreads, bs.smem_bytes, stream);
    if (e != cudaSuccess)
        return noalloc_fail(TIDE_ERR_CUDA, "fold launch: %s", cudaGetErrorString(e));
    tide::g_launches.fetch_add(1);
    return TIDE_OK;
}

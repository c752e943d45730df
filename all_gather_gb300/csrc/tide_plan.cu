// Host side of libtide: plan geometry (TIDE paper, Section 2.1), validation,
// device tables, and the C-ABI entry points declared in include/tide.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "tide_internal.h"

namespace tide {
std::atomic<uint64_t> g_launches{0};
}

namespace {

// Detail of the last failing call on this thread: a fixed buffer, so that
// reporting a failure never allocates (or throws).
thread_local char t_last_error[512];

tide_status_t fail(tide_status_t st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
tide_status_t fail(tide_status_t st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return st;
}

// Run a C-ABI body so that no C++ exception crosses the ABI: host
// allocation failures become TIDE_ERR_OOM.
template <typename F>
tide_status_t guarded(F &&body)
{
    try {
        return body();
    } catch (const std::bad_alloc &) {
        return fail(TIDE_ERR_OOM, "host memory allocation failed");
    } catch (...) {
        return fail(TIDE_ERR_INVALID_ARG, "unexpected internal error");
    }
}

tide_status_t cuda_fail(cudaError_t e, const char *what)
{
    return fail(TIDE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int64_t kMaxElems = int64_t(1) << 60;

bool mul_ok(int64_t a, int64_t b, int64_t *out)
{
    if (a < 0 || b < 0)
        return false;
    if (a != 0 && b > kMaxElems / a)
        return false;
    *out = a * b;
    return true;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Source phase of a piece: (address / 2) mod 8 of rank u's first element when
// every rank agrees, else -1 (the fold then uses scalar loads for it).
int32_t piece_phase(const uint64_t *ptrs_p, int32_t W, int64_t src_elem, int elem_bytes)
{
    const int shift = elem_bytes == 4 ? 2 : 1;
    const uint64_t mask = uint64_t(16 / elem_bytes - 1);
    int32_t ph = -1;
    for (int32_t u = 0; u < W; ++u) {
        int32_t x = int32_t(((ptrs_p[u] >> shift) + uint64_t(src_elem)) & mask);
        if (u == 0)
            ph = x;
        else if (x != ph)
            return -1;
    }
    return ph;
}

tide_status_t check_flags(const tide_plan_flags_t &f)
{
    if (f.reserved[0] != 0)
        return fail(TIDE_ERR_INVALID_ARG, "flags.reserved[0] must be zero");
    if (f.ce_streams < 0 || f.ce_streams > 8)
        return fail(TIDE_ERR_INVALID_ARG, "flags.ce_streams %d outside [0, 8]", f.ce_streams);
    if (f.fill_bytes != 0 && (f.fill_bytes < 16 || f.fill_bytes % 16 != 0 || f.fill_bytes > 16384))
        return fail(TIDE_ERR_INVALID_ARG, "flags.fill_bytes %d: need 0 or a multiple of 16 in [16, 16384]",
                    f.fill_bytes);
    if (f.fill_ranks < 0 || f.fill_ranks > tide::kMaxWorld)
        return fail(TIDE_ERR_INVALID_ARG, "flags.fill_ranks %d", f.fill_ranks);
    if (f.cta_budget < 0)
        return fail(TIDE_ERR_INVALID_ARG, "flags.cta_budget %d < 0", f.cta_budget);
    if (f.chunk_bytes != 0 && (f.chunk_bytes < 256 || f.chunk_bytes % 256 != 0 || f.chunk_bytes > (1 << 26)))
        return fail(TIDE_ERR_INVALID_ARG, "flags.chunk_bytes %d: need 0 or a multiple of 256 in [256, 2^26]",
                    f.chunk_bytes);
    if (f.order != TIDE_ORDER_RANK_ASC && f.order != TIDE_ORDER_STAGED_OWN && f.order != TIDE_ORDER_NODES &&
        f.order != TIDE_ORDER_TREE)
        return fail(TIDE_ERR_UNSUPPORTED, "flags.order %d is not implemented", f.order);
    if (f.order == TIDE_ORDER_NODES ? f.node_size < 1 : f.node_size != 0)
        return fail(TIDE_ERR_INVALID_ARG, "flags.node_size %d (positive with TIDE_ORDER_NODES only)", f.node_size);
    if (f.sched != TIDE_SCHED_AUTO && f.sched != TIDE_SCHED_STATIC && f.sched != TIDE_SCHED_DYNAMIC &&
        f.sched != TIDE_SCHED_PER_ITEM)
        return fail(TIDE_ERR_INVALID_ARG, "flags.sched %d", f.sched);
    if (f.sched == TIDE_SCHED_PER_ITEM && f.cta_budget != 0)
        return fail(TIDE_ERR_INVALID_ARG, "TIDE_SCHED_PER_ITEM sizes the grid itself: cta_budget must be 0");
    if (f.kernel != TIDE_KERNEL_AUTO && f.kernel != TIDE_KERNEL_DIRECT && f.kernel != TIDE_KERNEL_BULK)
        return fail(TIDE_ERR_INVALID_ARG, "flags.kernel %d", f.kernel);
    if (f.grad_dtype != TIDE_DTYPE_BF16 && f.grad_dtype != TIDE_DTYPE_F32)
        return fail(TIDE_ERR_UNSUPPORTED, "flags.grad_dtype %d is not implemented", f.grad_dtype);
    if ((f.order != TIDE_ORDER_RANK_ASC || f.grad_dtype != TIDE_DTYPE_BF16) && f.kernel == TIDE_KERNEL_DIRECT)
        return fail(TIDE_ERR_UNSUPPORTED, "orders other than rank order and fp32 gradients run on the bulk kernel");
    if (f.debug & ~(TIDE_DEBUG_HOST_ONLY | TIDE_DEBUG_SHORT_WAIT | TIDE_DEBUG_SKIP_FILL))
        return fail(TIDE_ERR_INVALID_ARG, "unknown debug bits 0x%x", f.debug);
    if ((f.debug & TIDE_DEBUG_SKIP_FILL) && f.kernel != TIDE_KERNEL_BULK)
        return fail(TIDE_ERR_INVALID_ARG, "TIDE_DEBUG_SKIP_FILL applies to the bulk-copy kernel only");
    return TIDE_OK;
}

// Copy and check the gradient pointers of every parameter into plan->ptrs and
// recompute each piece's source phase and the address hull.
tide_status_t load_pointers(tide_plan_t *plan, const tide_param_desc_t *params)
{
    const int32_t W = plan->world;
    uintptr_t lo = UINTPTR_MAX, hi = 0;
    for (int32_t p = 0; p < plan->nparams; ++p) {
        const int64_t numel = plan->dim0[p] * plan->row_numel[p];
        if (params[p].rank_base == nullptr)
            return fail(TIDE_ERR_INVALID_ARG, "params[%d].rank_base is NULL", p);
        for (int32_t u = 0; u < W; ++u) {
            uintptr_t a = reinterpret_cast<uintptr_t>(params[p].rank_base[u]);
            if (numel > 0 && a == 0)
                return fail(TIDE_ERR_INVALID_ARG, "params[%d].rank_base[%d] is NULL", p, u);
            if (a & uintptr_t(plan->elem_bytes - 1))
                return fail(TIDE_ERR_ALIGNMENT, "params[%d].rank_base[%d] is not %d-byte aligned", p, u,
                            plan->elem_bytes);
            plan->ptrs[size_t(p) * W + u] = a;
            if (numel > 0) {
                lo = std::min(lo, a);
                hi = std::max(hi, a + uintptr_t(numel) * uintptr_t(plan->elem_bytes));
            }
        }
    }
    plan->src_lo = lo;
    plan->src_hi = hi;
    for (auto &s : plan->segs)
        s.src_phase = piece_phase(&plan->ptrs[size_t(s.param) * W], W, s.src_elem, plan->elem_bytes);
    return TIDE_OK;
}

// Where the gradients live.  Device memory of the plan's device and managed
// memory are read by either kernel; page-locked host memory mapped into the
// device's address space is read in place over the host link (NVLink-C2C on
// Grace systems) by the direct-load kernel, whose plain loads reach it (the
// bulk-copy kernel is not used on host memory); pageable host memory cannot
// be read by a kernel and is refused.  kinds[i] = 1 for host memory; *host:
// some gradient is host memory.  A pointer equal to prev[i] keeps
// prev_kinds[i] without a query (a rebind to the same buffers costs nothing).
tide_status_t classify_gradients(const tide_plan_t *plan, bool *host, std::vector<uint8_t> &kinds,
                                 const std::vector<uint64_t> *prev = nullptr,
                                 const std::vector<uint8_t> *prev_kinds = nullptr)
{
    *host = false;
    kinds.assign(plan->ptrs.size(), 0);
    for (int32_t p = 0; p < plan->nparams; ++p) {
        if (plan->dim0[p] * plan->row_numel[p] == 0)
            continue;
        for (int32_t u = 0; u < plan->world; ++u) {
            const size_t i = size_t(p) * plan->world + u;
            if (prev && prev_kinds && prev_kinds->size() == kinds.size() && (*prev)[i] == plan->ptrs[i]) {
                kinds[i] = (*prev_kinds)[i];
                *host = *host || kinds[i];
                continue;
            }
            void *ptr = reinterpret_cast<void *>(plan->ptrs[i]);
            cudaPointerAttributes a{};
            cudaError_t e = cudaPointerGetAttributes(&a, ptr);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(TIDE_ERR_INVALID_ARG, "params[%d].rank_base[%d]: %s", p, u, cudaGetErrorString(e));
            }
            if (a.type == cudaMemoryTypeHost) {
                if (a.devicePointer != ptr)
                    return fail(TIDE_ERR_INVALID_ARG,
                                "params[%d].rank_base[%d] is page-locked host memory not mapped at the same address "
                                "on the device",
                                p, u);
                kinds[i] = 1;
                *host = true;
            } else if (a.type == cudaMemoryTypeDevice) {
                if (a.device != plan->device)
                    return fail(TIDE_ERR_INVALID_ARG, "params[%d].rank_base[%d] is memory of device %d, not %d", p, u,
                                a.device, plan->device);
            } else if (a.type != cudaMemoryTypeManaged) {
                return fail(TIDE_ERR_INVALID_ARG,
                            "params[%d].rank_base[%d] is pageable host memory: a kernel cannot read it "
                            "(use device, managed or page-locked host memory)",
                            p, u);
            }
        }
    }
    return TIDE_OK;
}

bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// Does [lo, hi) overlap any gradient tensor of the plan?
bool overlaps_gradients(const tide_plan_t *plan, uintptr_t lo, uintptr_t hi)
{
    if (lo >= hi || !ranges_overlap(lo, hi, plan->src_lo, plan->src_hi))
        return false;
    for (int32_t p = 0; p < plan->nparams; ++p) {
        const uintptr_t bytes = uintptr_t(plan->dim0[p] * plan->row_numel[p]) * uintptr_t(plan->elem_bytes);
        for (int32_t u = 0; u < plan->world; ++u) {
            uintptr_t a = plan->ptrs[size_t(p) * plan->world + u];
            if (bytes && ranges_overlap(lo, hi, a, a + bytes))
                return true;
        }
    }
    return false;
}

// Record the plan's last-use event on `stream`, except while the stream is
// being captured into a CUDA graph: a captured record would not mark a real
// point of execution, so destroy() synchronises the device instead (below).
cudaError_t mark_use(tide_plan_t *plan, cudaStream_t stream)
{
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess)
        return e;
    if (cap != cudaStreamCaptureStatusNone) {
        plan->captured = true;
        return cudaSuccess;
    }
    return cudaEventRecord(plan->last_use, stream);
}

tide_status_t upload_tables(tide_plan_t *plan, cudaStream_t stream, bool pointers_only)
{
    cudaError_t e;
    if (!pointers_only) {
        e = cudaMemcpyAsync(plan->d_rs_items, plan->rs_items.data(), plan->rs_items.size() * sizeof(tide::Item),
                            cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "upload work items");
        e = cudaMemcpyAsync(plan->d_ag_items, plan->ag_items.data(), plan->ag_items.size() * sizeof(tide::Item),
                            cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "upload placement items");
    }
    e = cudaMemcpyAsync(plan->d_ptrs, plan->ptrs.data(), plan->ptrs.size() * sizeof(uint64_t),
                        cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "upload pointer table");
    e = cudaMemcpyAsync(plan->d_segs, plan->segs.data(), plan->segs.size() * sizeof(tide::Seg),
                        cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "upload segment table");
    e = mark_use(plan, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "record plan event");
    return TIDE_OK;
}

void free_device(tide_plan_t *plan)
{
    if (plan->last_use) {
        cudaEventSynchronize(plan->last_use);
        cudaEventDestroy(plan->last_use);
        plan->last_use = nullptr;
    }
    if (plan->captured)  // graphs may still replay launches that read the tables
        cudaDeviceSynchronize();
    for (int i = 0; i < plan->n_ce; ++i) {
        cudaStreamSynchronize(plan->ce_stream[i]);
        cudaStreamDestroy(plan->ce_stream[i]);
        cudaEventDestroy(plan->ce_join[i]);
    }
    plan->n_ce = 0;
    if (plan->ce_fork) {
        cudaEventDestroy(plan->ce_fork);
        plan->ce_fork = nullptr;
    }
    if (plan->d_block) {
        cudaFree(plan->d_block);
        plan->d_block = nullptr;
    }
}

tide_status_t check_device(const tide_plan_t *plan)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev != plan->device)
        return fail(TIDE_ERR_INVALID_ARG, "plan was built on device %d but device %d is current", plan->device, dev);
    return TIDE_OK;
}

}  // namespace

extern "C" {

const char *tide_status_string(tide_status_t s)
{
    switch (s) {
    case TIDE_OK: return "TIDE_OK";
    case TIDE_ERR_INVALID_ARG: return "TIDE_ERR_INVALID_ARG";
    case TIDE_ERR_ALIGNMENT: return "TIDE_ERR_ALIGNMENT";
    case TIDE_ERR_UNSUPPORTED: return "TIDE_ERR_UNSUPPORTED";
    case TIDE_ERR_OOM: return "TIDE_ERR_OOM";
    case TIDE_ERR_CUDA: return "TIDE_ERR_CUDA";
    case TIDE_ERR_TIMEOUT: return "TIDE_ERR_TIMEOUT";
    }
    return "TIDE_ERR_UNKNOWN";
}

const char *tide_last_error(void) { return t_last_error; }

uint64_t tide_launch_count(void) { return tide::g_launches.load(); }

static tide_status_t plan_build_impl(int32_t world, int32_t num_params, const tide_param_desc_t *params,
                              const tide_plan_flags_t *flags, void *stream_, tide_plan_t **plan_out)
{
    t_last_error[0] = '\0';
    if (!plan_out)
        return fail(TIDE_ERR_INVALID_ARG, "plan_out is NULL");
    *plan_out = nullptr;
    if (world < 1 || world > tide::kMaxWorld)
        return fail(TIDE_ERR_INVALID_ARG, "world %d outside [1, %d]", world, tide::kMaxWorld);
    if (num_params < 0)
        return fail(TIDE_ERR_INVALID_ARG, "num_params %d < 0", num_params);
    if (num_params > 0 && !params)
        return fail(TIDE_ERR_INVALID_ARG, "params is NULL");
    tide_plan_flags_t f{};
    if (flags)
        f = *flags;
    tide_status_t st = check_flags(f);
    if (st != TIDE_OK)
        return st;

    auto *plan = new (std::nothrow) tide_plan_t();
    if (!plan)
        return fail(TIDE_ERR_OOM, "host allocation of the plan failed");
    auto bail = [&](tide_status_t s) {
        free_device(plan);
        delete plan;
        return s;
    };
    // The default schedule: dynamic claims (2-6% faster than the static split
    // on the benchmark groups), or static when every CTA gets at most one
    // work item (then a claim only adds latency); settled once the grid is known.
    const bool auto_sched = f.sched == TIDE_SCHED_AUTO;
    if (auto_sched)
        f.sched = TIDE_SCHED_DYNAMIC;
    plan->world = world;
    plan->nparams = num_params;
    plan->flags = f;
    plan->host_only = (f.debug & TIDE_DEBUG_HOST_ONLY) != 0;
    plan->chunk_elems = (f.chunk_bytes ? f.chunk_bytes : tide::kDefaultChunkBytes) / 2;
    plan->kernel = f.kernel == TIDE_KERNEL_AUTO ? TIDE_KERNEL_BULK : f.kernel;
    plan->elem_bytes = f.grad_dtype == TIDE_DTYPE_F32 ? 4 : 2;
    if (f.order == TIDE_ORDER_NODES && world % f.node_size != 0)
        return bail(fail(TIDE_ERR_INVALID_ARG, "node_size %d does not divide world %d", f.node_size, world));
    if (f.order == TIDE_ORDER_TREE) {
        const tide::BulkShape bs =
            tide::bulk_shape(world, f.fill_bytes / plan->elem_bytes, f.fill_ranks, false, plan->elem_bytes, f.order);
        if (world / bs.fill_ranks >= (1 << tide::kTreeLevels))
            return bail(fail(TIDE_ERR_INVALID_ARG,
                             "tree order: %d full stage fills of %d ranks per chunk (at most %d); raise fill_ranks",
                             world / bs.fill_ranks, bs.fill_ranks, (1 << tide::kTreeLevels) - 1));
    }

    // --- geometry (Section 2.1): R_p = ceil(D_p / W), o_p, S -------------
    plan->dim0.resize(num_params);
    plan->row_numel.resize(num_params);
    plan->rows.resize(num_params);
    plan->offset.resize(num_params);
    int64_t running = 0, S = 0;
    for (int32_t p = 0; p < num_params; ++p) {
        const int64_t D = params[p].dim0, K = params[p].row_numel;
        int64_t numel, piece, span;
        if (D < 0 || K < 0)
            return bail(fail(TIDE_ERR_INVALID_ARG, "params[%d]: dim0 %lld, row_numel %lld", p, (long long)D,
                             (long long)K));
        const int64_t R = (D + world - 1) / world;
        if (!mul_ok(D, K, &numel) || !mul_ok(R, K, &piece) || !mul_ok(piece, world, &span))
            return bail(fail(TIDE_ERR_INVALID_ARG, "params[%d]: size overflows", p));
        int64_t o = params[p].shard_offset;
        if (o < -1)
            return bail(fail(TIDE_ERR_INVALID_ARG, "params[%d].shard_offset %lld", p, (long long)o));
        if (o == -1)
            o = running;
        if (o > kMaxElems - piece)
            return bail(fail(TIDE_ERR_INVALID_ARG, "params[%d]: offset overflows", p));
        plan->dim0[p] = D;
        plan->row_numel[p] = K;
        plan->rows[p] = R;
        plan->offset[p] = o;
        running = o + piece;
        S = std::max(S, running);
    }
    {   // explicit offsets must not make shards overlap
        std::vector<std::pair<int64_t, int64_t>> iv;
        for (int32_t p = 0; p < num_params; ++p)
            if (plan->rows[p] * plan->row_numel[p] > 0)
                iv.emplace_back(plan->offset[p], plan->offset[p] + plan->rows[p] * plan->row_numel[p]);
        std::sort(iv.begin(), iv.end());
        for (size_t i = 1; i < iv.size(); ++i)
            if (iv[i].first < iv[i - 1].second)
                return bail(fail(TIDE_ERR_INVALID_ARG, "shard offsets make two parameters overlap in the slot"));
    }
    plan->slot_numel = S;
    int64_t total;
    if (!mul_ok(S, world, &total))
        return bail(fail(TIDE_ERR_INVALID_ARG, "W * S overflows"));

    // --- pieces: rank r owns rows [r R_p, (r+1) R_p), v = clamp(D - r R, 0, R)
    plan->segs.reserve(size_t(num_params) * world);
    for (int32_t p = 0; p < num_params; ++p) {
        const int64_t D = plan->dim0[p], K = plan->row_numel[p], R = plan->rows[p];
        for (int32_t r = 0; r < world; ++r) {
            int64_t v = std::min(std::max(D - int64_t(r) * R, int64_t(0)), R);
            tide::Seg s{};
            s.src_elem = int64_t(r) * R * K;
            s.dst_elem = plan->offset[p];
            s.n_valid = v * K;
            s.n_pad = (R - v) * K;
            s.param = p;
            s.rank = r;
            s.src_phase = -1;
            plan->segs.push_back(s);
        }
    }
    plan->ptrs.assign(size_t(num_params) * world, 0);
    st = load_pointers(plan, params);
    if (st != TIDE_OK)
        return bail(st);

    // --- work lists --------------------------------------------------------
    const int64_t CH = plan->chunk_elems;
    for (size_t i = 0; i < plan->segs.size(); ++i) {
        const tide::Seg &s = plan->segs[i];
        for (int64_t b = 0; b < s.n_valid; b += CH)
            plan->rs_items.push_back({int32_t(i), uint32_t(std::min(CH, s.n_valid - b)), b});
        for (int64_t b = 0; b < s.n_pad; b += CH)
            plan->rs_items.push_back({int32_t(i), uint32_t(std::min(CH, s.n_pad - b)) | tide::kItemPad, b});
    }
    plan->ag_param_item_begin.assign(size_t(num_params) + 1, 0);
    for (size_t i = 0; i < plan->segs.size(); ++i) {
        const tide::Seg &s = plan->segs[i];
        if (s.rank == 0)
            plan->ag_param_item_begin[s.param] = int64_t(plan->ag_items.size());
        for (int64_t b = 0; b < s.n_valid; b += tide::kAgChunkElems)
            plan->ag_items.push_back({int32_t(i), uint32_t(std::min(tide::kAgChunkElems, s.n_valid - b)), b});
    }
    plan->ag_param_item_begin[num_params] = int64_t(plan->ag_items.size());
    if (plan->segs.size() > size_t(INT32_MAX) || plan->rs_items.size() > size_t(INT32_MAX))
        return bail(fail(TIDE_ERR_UNSUPPORTED, "too many work items; raise chunk_bytes"));

    plan->block = plan->kernel == TIDE_KERNEL_BULK ? tide::kBulkThreads : tide::kFoldThreads;
    plan->fold_smem = tide::fold_smem_bytes(plan->kernel, world, f.fill_bytes / plan->elem_bytes, f.fill_ranks,
                                            false, plan->elem_bytes, f.order);
    if (plan->host_only) {
        plan->grid = f.sched == TIDE_SCHED_PER_ITEM ? int32_t(plan->rs_items.size()) : f.cta_budget ? f.cta_budget : 0;
        *plan_out = plan;
        return TIDE_OK;
    }

    // --- device tables -----------------------------------------------------
    cudaError_t e = cudaGetDevice(&plan->device);
    if (e != cudaSuccess)
        return bail(cuda_fail(e, "cudaGetDevice"));
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, plan->device);
    if (e != cudaSuccess)
        return bail(cuda_fail(e, "query SM count"));
    plan->sms = sms;
    st = classify_gradients(plan, &plan->host_grads, plan->ptr_host);
    if (st != TIDE_OK)
        return bail(st);
    if (plan->host_grads) {
        if (f.kernel == TIDE_KERNEL_BULK || f.order != TIDE_ORDER_RANK_ASC || f.grad_dtype != TIDE_DTYPE_BF16)
            return bail(fail(TIDE_ERR_UNSUPPORTED,
                             "gradients in host memory are folded by the direct-load kernel (bf16, rank order)"));
        plan->kernel = TIDE_KERNEL_DIRECT;
        plan->block = tide::kFoldThreads;
        plan->fold_smem = tide::fold_smem_bytes(TIDE_KERNEL_DIRECT, world, 0, 0, false);
    }
    plan->whole_sm = plan->kernel == TIDE_KERNEL_BULK && f.cta_budget > 0 && f.cta_budget <= sms;
    if (plan->whole_sm)
        plan->fold_smem = tide::fold_smem_bytes(plan->kernel, world, f.fill_bytes / plan->elem_bytes, f.fill_ranks,
                                                true, plan->elem_bytes, f.order);
    plan->consumer_warps = tide::bulk_consumer_warps(plan->whole_sm, f.order, f.grad_dtype);
    if (plan->kernel == TIDE_KERNEL_BULK)
        plan->block = 32 * (1 + plan->consumer_warps);
    int per_sm = 0;
    e = tide::fold_occupancy(plan->kernel, world, plan->block, plan->fold_smem, &per_sm, f.grad_dtype, f.order,
                             f.fill_ranks, plan->consumer_warps);
    if (e != cudaSuccess)
        return bail(cuda_fail(e, "fold occupancy"));
    if (per_sm < 1)
        return bail(fail(TIDE_ERR_UNSUPPORTED, "fold kernel does not fit on an SM (world %d)", world));
    plan->grid = f.sched == TIDE_SCHED_PER_ITEM ? int32_t(std::max<size_t>(plan->rs_items.size(), 1))
                 : f.cta_budget ? f.cta_budget : sms * per_sm;
    if (auto_sched && int64_t(plan->rs_items.size()) <= int64_t(plan->grid))
        plan->flags.sched = TIDE_SCHED_STATIC;

    size_t off = 0;
    auto carve = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + std::max<size_t>(bytes, 1), 256);
        return at;
    };
    const size_t o_ptrs = carve(plan->ptrs.size() * sizeof(uint64_t));
    const size_t o_segs = carve(plan->segs.size() * sizeof(tide::Seg));
    const size_t o_rs = carve(plan->rs_items.size() * sizeof(tide::Item));
    const size_t o_ag = carve(plan->ag_items.size() * sizeof(tide::Item));
    const size_t o_cnt = carve(2 * sizeof(uint32_t));
    const size_t o_st = carve(sizeof(int32_t));
    e = cudaMalloc(&plan->d_block, off);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return bail(fail(TIDE_ERR_OOM, "cudaMalloc of %zu table bytes: %s", off, cudaGetErrorString(e)));
    }
    char *base = static_cast<char *>(plan->d_block);
    plan->d_ptrs = reinterpret_cast<uint64_t *>(base + o_ptrs);
    plan->d_segs = reinterpret_cast<tide::Seg *>(base + o_segs);
    plan->d_rs_items = reinterpret_cast<tide::Item *>(base + o_rs);
    plan->d_ag_items = reinterpret_cast<tide::Item *>(base + o_ag);
    plan->d_counters = reinterpret_cast<uint32_t *>(base + o_cnt);
    plan->d_status = reinterpret_cast<int32_t *>(base + o_st);
    e = cudaEventCreateWithFlags(&plan->last_use, cudaEventDisableTiming);
    if (e != cudaSuccess)
        return bail(cuda_fail(e, "create plan event"));
    e = cudaEventCreateWithFlags(&plan->ce_fork, cudaEventDisableTiming);
    if (e != cudaSuccess)
        return bail(cuda_fail(e, "create copy-engine event"));
    for (int i = 0, n = f.ce_streams ? f.ce_streams : 8; i < n; ++i) {
        e = cudaStreamCreateWithFlags(&plan->ce_stream[i], cudaStreamNonBlocking);
        if (e == cudaSuccess) {
            e = cudaEventCreateWithFlags(&plan->ce_join[i], cudaEventDisableTiming);
            if (e != cudaSuccess)
                cudaStreamDestroy(plan->ce_stream[i]);
        }
        if (e != cudaSuccess)
            return bail(cuda_fail(e, "create copy-engine stream"));
        plan->n_ce = i + 1;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    e = cudaMemsetAsync(base + o_cnt, 0, o_st + sizeof(int32_t) - o_cnt, stream);
    if (e != cudaSuccess)
        return bail(cuda_fail(e, "clear counters"));
    st = upload_tables(plan, stream, false);
    if (st != TIDE_OK)
        return bail(st);
    *plan_out = plan;
    return TIDE_OK;
}

static tide_status_t plan_rebind_impl(tide_plan_t *plan, const tide_param_desc_t *params, void *stream)
{
    t_last_error[0] = '\0';
    if (!plan)
        return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
    if (plan->nparams > 0 && !params)
        return fail(TIDE_ERR_INVALID_ARG, "params is NULL");
    for (int32_t p = 0; p < plan->nparams; ++p) {
        const int64_t o = params[p].shard_offset;
        if (params[p].dim0 != plan->dim0[p] || params[p].row_numel != plan->row_numel[p] ||
            (o != -1 && o != plan->offset[p]))
            return fail(TIDE_ERR_INVALID_ARG, "params[%d] geometry differs from the plan's", p);
    }
    std::vector<uint64_t> keep_ptrs = plan->ptrs;
    std::vector<tide::Seg> keep_segs = plan->segs;
    uintptr_t keep_lo = plan->src_lo, keep_hi = plan->src_hi;
    tide_status_t st = load_pointers(plan, params);
    if (st != TIDE_OK) {
        plan->ptrs.swap(keep_ptrs);
        plan->segs.swap(keep_segs);
        plan->src_lo = keep_lo;
        plan->src_hi = keep_hi;
        return st;
    }
    if (plan->host_only)
        return TIDE_OK;
    st = check_device(plan);
    bool host = false;
    std::vector<uint8_t> kinds;
    if (st == TIDE_OK)
        st = classify_gradients(plan, &host, kinds, &keep_ptrs, &plan->ptr_host);
    if (st == TIDE_OK && host != plan->host_grads)
        st = fail(TIDE_ERR_INVALID_ARG, "rebind cannot move gradients between host and device memory");
    if (st == TIDE_OK)
        plan->ptr_host.swap(kinds);
    if (st != TIDE_OK) {
        plan->ptrs.swap(keep_ptrs);
        plan->segs.swap(keep_segs);
        plan->src_lo = keep_lo;
        plan->src_hi = keep_hi;
        return st;
    }
    return upload_tables(plan, static_cast<cudaStream_t>(stream), true);
}

tide_status_t tide_rs_fold(tide_plan_t *plan, float *out_base, int64_t out_slot_stride, float alpha,
                           int32_t accumulate, void *stream_)
{
    tide::NvtxRange range("tide_rs_fold");
    t_last_error[0] = '\0';
    if (!plan)
        return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
    if (plan->host_only)
        return fail(TIDE_ERR_INVALID_ARG, "plan was built host-only and cannot be launched");
    if (accumulate != 0 && accumulate != 1)
        return fail(TIDE_ERR_INVALID_ARG, "accumulate must be 0 or 1");
    if (out_slot_stride < plan->slot_numel)
        return fail(TIDE_ERR_INVALID_ARG, "out_slot_stride %lld < S %lld", (long long)out_slot_stride,
                    (long long)plan->slot_numel);
    if (plan->rs_items.empty())
        return TIDE_OK;
    if (!out_base)
        return fail(TIDE_ERR_INVALID_ARG, "out_base is NULL");
    if (reinterpret_cast<uintptr_t>(out_base) & 3u)
        return fail(TIDE_ERR_ALIGNMENT, "out_base is not 4-byte aligned");
    int64_t span;
    if (!mul_ok(out_slot_stride, plan->world - 1, &span) || span > kMaxElems - plan->slot_numel)
        return fail(TIDE_ERR_INVALID_ARG, "output extent overflows");
    const uintptr_t lo = reinterpret_cast<uintptr_t>(out_base);
    const uintptr_t hi = lo + uintptr_t(span + plan->slot_numel) * 4u;
    if (overlaps_gradients(plan, lo, hi))
        return fail(TIDE_ERR_INVALID_ARG, "the output overlaps a gradient tensor");
    tide_status_t st = check_device(plan);
    if (st != TIDE_OK)
        return st;

    tide::FoldParams fp{};
    fp.ptrs = plan->d_ptrs;
    fp.segs = plan->d_segs;
    fp.items = plan->d_rs_items;
    fp.n_items = int64_t(plan->rs_items.size());
    fp.out = out_base;
    fp.stride = out_slot_stride;
    fp.alpha = alpha;
    fp.world = plan->world;
    fp.sched = plan->flags.sched;
    fp.counters = plan->d_counters;
    fp.status = plan->d_status;
    fp.debug = plan->flags.debug;
    fp.wait_budget_ns = (plan->flags.debug & TIDE_DEBUG_SHORT_WAIT) ? tide::kShortWaitBudgetNs : tide::kWaitBudgetNs;
    const tide::BulkShape bs = tide::bulk_shape(plan->world, plan->flags.fill_bytes / plan->elem_bytes,
                                                plan->flags.fill_ranks, plan->whole_sm, plan->elem_bytes,
                                                plan->flags.order);
    fp.order = plan->flags.order;
    fp.node_size = plan->flags.node_size;
    fp.dtype = plan->flags.grad_dtype;
    fp.fill_elems = bs.fill_elems;
    fp.fill_ranks = bs.fill_ranks;
    fp.stages = bs.stages;
    fp.consumer_warps = plan->consumer_warps;
    const int grid = int(std::min<int64_t>(plan->grid, fp.n_items));
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    cudaError_t e = tide::launch_fold(fp, plan->kernel, accumulate, grid, plan->block, plan->fold_smem, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "fold launch");
    tide::g_launches.fetch_add(1);
    e = mark_use(plan, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "record plan event");
    return TIDE_OK;
}

}  // extern "C"

namespace {

// Common checks of both placements: plan, mode-independent sizes, the slot
// range [s_lo, s_hi) and the full[] tensors (non-null, aligned, disjoint from
// the slots and from each other).
tide_status_t check_placement(tide_plan_t *plan, const void *slots_base, int64_t slot_stride, size_t elem_bytes,
                              void *const *full)
{
    if (!plan)
        return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
    if (plan->host_only)
        return fail(TIDE_ERR_INVALID_ARG, "plan was built host-only and cannot be launched");
    if (slot_stride < plan->slot_numel)
        return fail(TIDE_ERR_INVALID_ARG, "slot_stride %lld < S %lld", (long long)slot_stride,
                    (long long)plan->slot_numel);
    if (plan->ag_items.empty())
        return TIDE_OK;
    if (!slots_base || !full)
        return fail(TIDE_ERR_INVALID_ARG, "slots_base or full is NULL");
    if (reinterpret_cast<uintptr_t>(slots_base) & (elem_bytes - 1))
        return fail(TIDE_ERR_ALIGNMENT, "slots_base is not %zu-byte aligned", elem_bytes);
    int64_t span;
    if (!mul_ok(slot_stride, plan->world - 1, &span) || span > kMaxElems - plan->slot_numel)
        return fail(TIDE_ERR_INVALID_ARG, "slot extent overflows");
    const uintptr_t s_lo = reinterpret_cast<uintptr_t>(slots_base);
    const uintptr_t s_hi = s_lo + uintptr_t(span + plan->slot_numel) * elem_bytes;
    std::vector<std::pair<uintptr_t, uintptr_t>> iv;
    iv.reserve(plan->nparams);
    for (int32_t p = 0; p < plan->nparams; ++p) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(full[p]);
        const uintptr_t bytes = uintptr_t(plan->dim0[p] * plan->row_numel[p]) * 2u;
        if (bytes == 0)
            continue;
        if (a == 0)
            return fail(TIDE_ERR_INVALID_ARG, "full[%d] is NULL", p);
        if (a & 1u)
            return fail(TIDE_ERR_ALIGNMENT, "full[%d] is not 2-byte aligned", p);
        if (ranges_overlap(a, a + bytes, s_lo, s_hi))
            return fail(TIDE_ERR_INVALID_ARG, "full[%d] overlaps the shard slots", p);
        iv.emplace_back(a, a + bytes);
    }
    std::sort(iv.begin(), iv.end());
    for (size_t i = 1; i < iv.size(); ++i)
        if (iv[i].first < iv[i - 1].second)
            return fail(TIDE_ERR_INVALID_ARG, "two full[] tensors overlap");
    return check_device(plan);
}

// Copy-engine placement.  Rank r's piece of p: slot r at o_p -> full_p rows
// [r R, r R + v).  As 2D copies, one per parameter over the ranks holding R
// real rows (source pitch = slot stride, destination pitch = R K) plus one
// tail copy, or as one 1D copy per piece.  Pieces of kCeRowCopyBytes or more
// are copied one by one even in 2D mode: they need few descriptors, and the
// copy engines move large 1D copies faster than 2D ones.  The copies are spread over the
// plan's internal streams so that several copy engines work at once: large
// 2D copies are split by rows, then each copy goes to the least loaded
// stream.  The internal streams fork from and join back into `stream`.
constexpr size_t kCeRowCopyBytes = size_t(1) << 20;

struct CeCopy {
    char *dst;
    size_t dpitch;
    const char *src;
    size_t spitch, width, height;
};

tide_status_t copy_engine_placement(tide_plan_t *plan, const uint16_t *slots, int64_t slot_stride, void *const *full,
                                    bool two_d, cudaStream_t stream)
{
    std::vector<CeCopy> jobs;
    size_t total = 0;
    for (int32_t p = 0; p < plan->nparams; ++p) {
        const int64_t D = plan->dim0[p], K = plan->row_numel[p], R = plan->rows[p];
        if (D * K == 0)
            continue;
        char *dst = static_cast<char *>(full[p]);
        const char *src = reinterpret_cast<const char *>(slots + plan->offset[p]);
        const size_t piece = size_t(R * K) * 2u, spitch = size_t(slot_stride) * 2u;
        const int64_t nfull = D / R;  // ranks holding R real rows
        if (two_d && nfull > 0 && piece < kCeRowCopyBytes) {
            jobs.push_back({dst, piece, src, spitch, piece, size_t(nfull)});
        } else {
            for (int64_t r = 0; r < nfull; ++r)
                jobs.push_back({dst + size_t(r) * piece, piece, src + size_t(r) * spitch, spitch, piece, 1});
        }
        const int64_t tail_rows = D - nfull * R;
        if (tail_rows > 0)
            jobs.push_back({dst + size_t(nfull) * piece, piece, src + size_t(nfull) * spitch, spitch,
                            size_t(tail_rows * K) * 2u, 1});
        total += size_t(D * K) * 2u;
    }
    const int n = plan->n_ce;
    if (n > 1) {  // split large 2D copies by rows into pieces of about total / (2 n)
        const size_t target = std::max<size_t>(total / size_t(2 * n), 1);
        std::vector<CeCopy> split;
        for (const CeCopy &j : jobs) {
            const size_t bytes = j.width * j.height;
            size_t k = std::min(j.height, (bytes + target - 1) / target);
            if (k <= 1) {
                split.push_back(j);
                continue;
            }
            const size_t rows = (j.height + k - 1) / k;
            for (size_t r0 = 0; r0 < j.height; r0 += rows)
                split.push_back({j.dst + r0 * j.dpitch, j.dpitch, j.src + r0 * j.spitch, j.spitch, j.width,
                                 std::min(rows, j.height - r0)});
        }
        jobs.swap(split);
        std::stable_sort(jobs.begin(), jobs.end(),
                         [](const CeCopy &a, const CeCopy &b) { return a.width * a.height > b.width * b.height; });
    }
    cudaError_t e = cudaSuccess;
    if (n > 1) {
        e = cudaEventRecord(plan->ce_fork, stream);
        for (int i = 0; i < n && e == cudaSuccess; ++i)
            e = cudaStreamWaitEvent(plan->ce_stream[i], plan->ce_fork, 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "fork copy-engine streams");
    }
    std::vector<size_t> load(size_t(std::max(n, 1)), 0);
    for (const CeCopy &j : jobs) {
        size_t best = 0;
        for (size_t i = 1; i < load.size(); ++i)
            if (load[i] < load[best])
                best = i;
        load[best] += j.width * j.height;
        cudaStream_t s = n > 1 ? plan->ce_stream[best] : stream;
        e = j.height > 1 ? cudaMemcpy2DAsync(j.dst, j.dpitch, j.src, j.spitch, j.width, j.height,
                                             cudaMemcpyDeviceToDevice, s)
                         : cudaMemcpyAsync(j.dst, j.src, j.width, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "placement copy");
    }
    if (n > 1) {
        for (int i = 0; i < n && e == cudaSuccess; ++i) {
            e = cudaEventRecord(plan->ce_join[i], plan->ce_stream[i]);
            if (e == cudaSuccess)
                e = cudaStreamWaitEvent(stream, plan->ce_join[i], 0);
        }
        if (e != cudaSuccess)
            return cuda_fail(e, "join copy-engine streams");
    }
    return TIDE_OK;
}

// Placement kernel launches, at most kAgParamsPerLaunch destination pointers each.
tide_status_t launch_placement(tide_plan_t *plan, const uint16_t *slots, const float *slots_f32,
                               int64_t slot_stride, void *const *full, cudaStream_t stream)
{
    static thread_local tide::AgParams ap;  // ~8 KB: keep it off the stack
    for (int32_t p0 = 0; p0 < plan->nparams; p0 += tide::kAgParamsPerLaunch) {
        const int32_t p1 = std::min(plan->nparams, p0 + tide::kAgParamsPerLaunch);
        ap.segs = plan->d_segs;
        ap.items = plan->d_ag_items;
        ap.item_begin = plan->ag_param_item_begin[p0];
        ap.item_end = plan->ag_param_item_begin[p1];
        if (ap.item_end == ap.item_begin)
            continue;
        ap.slots = slots;
        ap.slots_f32 = slots_f32;
        ap.stride = slot_stride;
        ap.param_base = p0;
        ap.n_full = p1 - p0;
        for (int32_t p = p0; p < p1; ++p)
            ap.full[p - p0] = static_cast<uint16_t *>(full[p]);
        const int64_t n = ap.item_end - ap.item_begin;
        // One short CTA per item: faster than a persistent grid on every
        // benchmark group (6.85 vs 6.66 TB/s on the Llama-8B block), and the
        // placement yields SMs to higher-priority work as its CTAs retire.
        const int grid = int(std::min<int64_t>(n, int64_t(INT32_MAX)));
        cudaError_t e = slots_f32 ? tide::launch_ag_f32(ap, grid, stream) : tide::launch_ag(ap, grid, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "placement launch");
        tide::g_launches.fetch_add(1);
    }
    return TIDE_OK;
}

}  // namespace

extern "C" {

static tide_status_t ag_place_impl(tide_plan_t *plan, const void *slots_base, int64_t slot_stride, void *const *full,
                            int32_t mode, void *stream_)
{
    t_last_error[0] = '\0';
    if (mode != TIDE_AG_SM && mode != TIDE_AG_CE_2D && mode != TIDE_AG_CE_1D)
        return fail(TIDE_ERR_INVALID_ARG, "unknown placement mode %d", mode);
    tide_status_t st = check_placement(plan, slots_base, slot_stride, 2, full);
    if (st != TIDE_OK || plan->ag_items.empty())
        return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const auto *slots = static_cast<const uint16_t *>(slots_base);
    cudaError_t e = cudaSuccess;

    if (mode == TIDE_AG_SM) {
        st = launch_placement(plan, slots, nullptr, slot_stride, full, stream);
        if (st != TIDE_OK)
            return st;
    } else {
        st = copy_engine_placement(plan, slots, slot_stride, full, mode == TIDE_AG_CE_2D, stream);
        if (st != TIDE_OK)
            return st;
    }
    e = mark_use(plan, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "record plan event");
    return TIDE_OK;
}

static tide_status_t ag_place_f32_impl(tide_plan_t *plan, const float *slots_base, int64_t slot_stride, void *const *full,
                                void *stream_)
{
    t_last_error[0] = '\0';
    tide_status_t st = check_placement(plan, slots_base, slot_stride, 4, full);
    if (st != TIDE_OK || plan->ag_items.empty())
        return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    st = launch_placement(plan, nullptr, slots_base, slot_stride, full, stream);
    if (st != TIDE_OK)
        return st;
    cudaError_t e = mark_use(plan, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "record plan event");
    return TIDE_OK;
}

tide_status_t tide_plan_destroy(tide_plan_t *plan)
{
    t_last_error[0] = '\0';
    if (!plan)
        return TIDE_OK;
    free_device(plan);
    delete plan;
    return TIDE_OK;
}

int64_t tide_plan_slot_numel(const tide_plan_t *plan) { return plan ? plan->slot_numel : -1; }

int64_t tide_plan_num_segments(const tide_plan_t *plan) { return plan ? int64_t(plan->segs.size()) : -1; }

tide_status_t tide_plan_segment(const tide_plan_t *plan, int64_t index, tide_segment_t *out)
{
    if (!plan || !out)
        return fail(TIDE_ERR_INVALID_ARG, "plan or out is NULL");
    if (index < 0 || index >= int64_t(plan->segs.size()))
        return fail(TIDE_ERR_INVALID_ARG, "segment index %lld out of range", (long long)index);
    const tide::Seg &s = plan->segs[size_t(index)];
    out->param = s.param;
    out->rank = s.rank;
    out->src_elem = s.src_elem;
    out->dst_elem = s.dst_elem;
    out->n_valid = s.n_valid;
    out->n_pad = s.n_pad;
    return TIDE_OK;
}

tide_status_t tide_plan_fold_config(const tide_plan_t *plan, int32_t *grid, int32_t *block, int64_t *items,
                                    int64_t *chunk_elems)
{
    if (!plan)
        return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
    const int64_t n = int64_t(plan->rs_items.size());
    if (grid)
        *grid = int32_t(std::min<int64_t>(plan->grid, n));
    if (block)
        *block = plan->block;
    if (items)
        *items = n;
    if (chunk_elems)
        *chunk_elems = plan->chunk_elems;
    return TIDE_OK;
}

tide_status_t tide_last_device_status(tide_plan_t *plan, void *stream_)
{
    t_last_error[0] = '\0';
    int32_t *status = nullptr;
    if (plan) {
        if (plan->host_only)
            return TIDE_OK;
        status = plan->d_status;
    } else {  // the allocation-free fold's status word on the current device
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetDevice");
        status = tide::noalloc_status_word(dev);
        if (!status)
            return TIDE_OK;  // that entry point never ran on this device
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, status, sizeof word, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "read device status");
    if (word != 0) {
        e = cudaMemsetAsync(status, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "clear device status");
        return fail(TIDE_ERR_TIMEOUT, "a bounded device wait expired (code %d)", word);
    }
    return TIDE_OK;
}

}  // extern "C"

namespace tide {
void record_error(const char *msg) { snprintf(t_last_error, sizeof t_last_error, "%s", msg); }
}  // namespace tide

// C-ABI entry points whose bodies allocate host memory: no exception escapes.
extern "C" {

tide_status_t tide_plan_build(int32_t world, int32_t num_params, const tide_param_desc_t *params,
                              const tide_plan_flags_t *flags, void *stream, tide_plan_t **plan_out)
{
    tide::NvtxRange range("tide_plan_build");
    return guarded([&] { return plan_build_impl(world, num_params, params, flags, stream, plan_out); });
}

tide_status_t tide_plan_rebind(tide_plan_t *plan, const tide_param_desc_t *params, void *stream)
{
    return guarded([&] { return plan_rebind_impl(plan, params, stream); });
}

tide_status_t tide_ag_place(tide_plan_t *plan, const void *slots_base, int64_t slot_stride, void *const *full,
                            int32_t mode, void *stream)
{
    tide::NvtxRange range("tide_ag_place");
    return guarded([&] { return ag_place_impl(plan, slots_base, slot_stride, full, mode, stream); });
}

tide_status_t tide_ag_place_f32(tide_plan_t *plan, const float *slots_base, int64_t slot_stride, void *const *full,
                                void *stream)
{
    tide::NvtxRange range("tide_ag_place_f32");
    return guarded([&] { return ag_place_f32_impl(plan, slots_base, slot_stride, full, stream); });
}

}  // extern "C"

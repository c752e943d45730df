// Reduce-scatter fold kernels: TIDE paper Section 4, Equation (5), with every
// one of the W ranks virtual (all gradient sets in this GPU's memory).
//
// For every (parameter p, rank r) piece and every element j of it:
//     acc  = f32(G_p^(0)[r R_p K_p + j])
//     acc  = acc + f32(G_p^(u)[...])   for u = 1 .. W-1    (fp32, RN, rank order)
//     y    = alpha * acc
//     out[r * stride + o_p + j] = accumulate ? out_old + y : y
// and for padding positions (rows past D_p) the same with zero contributions.
// (Section 4.3's other orders permute or group the additions, see seq_rank;
// the tree order adds them pairwise, see tree_push.)
//
// The work is HBM-bound (W bf16 reads + one fp32 write, +1 fp32 read when
// accumulating, per output element; ~0.4 flop/byte), so both kernels are
// built around bytes in flight.  One persistent grid walks the plan's work
// list of (piece, chunk) items, reading every rank's rows in place from the
// gradients' own storage (no pack buffer):
//   fold_bulk_kernel (default): one producer lane per CTA stages the rank rows
//     in a shared-memory ring with bulk asynchronous copies (the TMA engine),
//     four consumer warps add them in fp32 registers and store the shard;
//     the producer claims work items from a device counter and posts them to
//     the consumers (dynamic schedule), or takes every gridDim-th item;
//   fold_direct_kernel: every thread loads 16-byte vectors of the rank rows
//     straight into registers (static or dynamic item scheduling); the kernel
//     for gradients in page-locked host memory.
#include <cuda_runtime.h>

#include "tide_internal.h"

namespace tide {
namespace {

// 16 bytes of read-once gradient data: non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const uint16_t *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_bf16(const uint16_t *p)
{
    unsigned short v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return __uint_as_float(uint32_t(v) << 16);
}

// bf16 -> fp32 is exact: a bf16 is the upper half of a binary32.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 &x, float (&f)[8])
{
    f[0] = bf_lo(x.x); f[1] = bf_hi(x.x);
    f[2] = bf_lo(x.y); f[3] = bf_hi(x.y);
    f[4] = bf_lo(x.z); f[5] = bf_hi(x.z);
    f[6] = bf_lo(x.w); f[7] = bf_hi(x.w);
}

template <bool ACC>
__device__ __forceinline__ void store8(float *d, const float (&acc)[8], float alpha, bool vec)
{
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        y[e] = __fmul_rn(alpha, acc[e]);
    if (vec) {
        float4 *d4 = reinterpret_cast<float4 *>(d);
        if (ACC) {
            const float4 o0 = __ldcs(d4), o1 = __ldcs(d4 + 1);
            y[0] = __fadd_rn(o0.x, y[0]); y[1] = __fadd_rn(o0.y, y[1]);
            y[2] = __fadd_rn(o0.z, y[2]); y[3] = __fadd_rn(o0.w, y[3]);
            y[4] = __fadd_rn(o1.x, y[4]); y[5] = __fadd_rn(o1.y, y[5]);
            y[6] = __fadd_rn(o1.z, y[6]); y[7] = __fadd_rn(o1.w, y[7]);
        }
        __stcs(d4, make_float4(y[0], y[1], y[2], y[3]));
        __stcs(d4 + 1, make_float4(y[4], y[5], y[6], y[7]));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float v = y[e];
            if (ACC)
                v = __fadd_rn(d[e], v);
            __stcs(d + e, v);
        }
    }
}

__device__ __forceinline__ void load8(const float *d, float (&o)[8], bool vec)
{
    if (vec) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(d));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(d) + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            o[e] = __ldcs(d + e);
    }
}

// y = alpha * acc, then old + y when accumulating (old already loaded).
template <bool ACC>
__device__ __forceinline__ void store8_onto(float *d, const float (&acc)[8], const float (&old)[8], float alpha,
                                            bool vec)
{
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        y[e] = __fmul_rn(alpha, acc[e]);
        if (ACC)
            y[e] = __fadd_rn(old[e], y[e]);
    }
    if (vec) {
        float4 *d4 = reinterpret_cast<float4 *>(d);
        __stcs(d4, make_float4(y[0], y[1], y[2], y[3]));
        __stcs(d4 + 1, make_float4(y[4], y[5], y[6], y[7]));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            __stcs(d + e, y[e]);
    }
}

// One element by scalar loads (misaligned heads, tails and pieces).
template <int WT, bool ACC>
__device__ __forceinline__ void fold_scalar(const uint64_t *s_src, int W, int64_t e, float *dst, float alpha)
{
    float acc = ld_bf16(reinterpret_cast<const uint16_t *>(s_src[0]) + e);
#pragma unroll 4
    for (int u = 1; u < (WT > 0 ? WT : W); ++u)
        acc = __fadd_rn(acc, ld_bf16(reinterpret_cast<const uint16_t *>(s_src[u]) + e));
    float y = __fmul_rn(alpha, acc);
    if (ACC)
        y = __fadd_rn(dst[e], y);
    __stcs(dst + e, y);
}

// Padding rows: W zero contributions sum to +0, then scale / accumulate.
template <bool ACC>
__device__ void fold_pad(float *dst, int64_t count, float alpha)
{
    const float y = __fmul_rn(alpha, 0.0f);
    const int64_t mis = int64_t((reinterpret_cast<uintptr_t>(dst) >> 2) & 3u);
    int64_t head = (4 - mis) & 3;
    if (head > count)
        head = count;
    for (int64_t e = threadIdx.x; e < head; e += blockDim.x)
        __stcs(dst + e, ACC ? __fadd_rn(dst[e], y) : y);
    const int64_t nv = (count - head) >> 2;
    float4 *d4 = reinterpret_cast<float4 *>(dst + head);
    for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
        float4 o = make_float4(y, y, y, y);
        if (ACC) {
            const float4 p = __ldcs(d4 + v);
            o = make_float4(__fadd_rn(p.x, y), __fadd_rn(p.y, y), __fadd_rn(p.z, y), __fadd_rn(p.w, y));
        }
        __stcs(d4 + v, o);
    }
    for (int64_t e = head + nv * 4 + threadIdx.x; e < count; e += blockDim.x)
        __stcs(dst + e, ACC ? __fadd_rn(dst[e], y) : y);
}

// WT: compile-time world (0 = runtime).  G: ranks whose loads are issued
// together before their adds.  VPT: 8-element vectors per thread per pass.
template <int WT, int G, int VPT, bool ACC>
__global__ void __launch_bounds__(kFoldThreads) fold_direct_kernel(const FoldParams fp)
{
    extern __shared__ uint64_t s_src[];  // this item's W source pointers
    __shared__ int64_t s_next;
    const int W = WT > 0 ? WT : fp.world;
    const int tid = threadIdx.x;
    constexpr int NT = kFoldThreads;
    const float alpha = fp.alpha;
    const bool dynamic = fp.sched == TIDE_SCHED_DYNAMIC;

    int64_t it;
    if (dynamic) {
        if (tid == 0)
            s_next = int64_t(atomicAdd(fp.counters, 1u));
        __syncthreads();
        it = s_next;
    } else {
        it = blockIdx.x;
    }

    while (it < fp.n_items) {
        const Item item = fp.items[it];
        const Seg seg = fp.segs[item.seg];
        const int64_t count = int64_t(item.count_kind & ~kItemPad);
        const bool pad = (item.count_kind & kItemPad) != 0;
        float *dst = fp.out + int64_t(seg.rank) * fp.stride + seg.dst_elem + (pad ? seg.n_valid : 0) + item.begin;

        if (pad) {
            fold_pad<ACC>(dst, count, alpha);
        } else {
            for (int u = tid; u < W; u += NT)
                s_src[u] = fp.ptrs[int64_t(seg.param) * W + u] + uint64_t(seg.src_elem + item.begin) * 2u;
            __syncthreads();
            if (seg.src_phase >= 0) {
                // Every rank's row starts at the same phase: after h scalar
                // elements all W sources are 16-byte aligned.
                int64_t h = (8 - seg.src_phase) & 7;
                if (h > count)
                    h = count;
                const int64_t nvec = (count - h) >> 3;
                float *dv = dst + h;
                const bool dst_vec = (reinterpret_cast<uintptr_t>(dv) & 15u) == 0;
                for (int64_t v = tid; v < nvec; v += int64_t(NT) * VPT) {
                    float acc[VPT][8];
#pragma unroll
                    for (int u0 = 0; u0 < (WT > 0 ? WT : W); u0 += G) {
                        uint4 x[G][VPT];
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            if (u0 + g < W) {
                                const uint16_t *sp = reinterpret_cast<const uint16_t *>(s_src[u0 + g]) + h;
#pragma unroll
                                for (int j = 0; j < VPT; ++j) {
                                    const int64_t vj = v + int64_t(j) * NT;
                                    x[g][j] = vj < nvec ? ld_stream_v4(sp + vj * 8) : make_uint4(0, 0, 0, 0);
                                }
                            }
                        }
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            if (u0 + g < W) {
#pragma unroll
                                for (int j = 0; j < VPT; ++j) {
                                    float f[8];
                                    unpack8(x[g][j], f);
                                    if (u0 + g == 0) {
#pragma unroll
                                        for (int e = 0; e < 8; ++e)
                                            acc[j][e] = f[e];
                                    } else {
#pragma unroll
                                        for (int e = 0; e < 8; ++e)
                                            acc[j][e] = __fadd_rn(acc[j][e], f[e]);
                                    }
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const int64_t vj = v + int64_t(j) * NT;
                        if (vj < nvec)
                            store8<ACC>(dv + vj * 8, acc[j], alpha, dst_vec);
                    }
                }
                for (int64_t e = tid; e < h; e += NT)
                    fold_scalar<WT, ACC>(s_src, W, e, dst, alpha);
                for (int64_t e = h + nvec * 8 + tid; e < count; e += NT)
                    fold_scalar<WT, ACC>(s_src, W, e, dst, alpha);
            } else {
                for (int64_t e = tid; e < count; e += NT)
                    fold_scalar<WT, ACC>(s_src, W, e, dst, alpha);
            }
        }
        __syncthreads();  // s_src / s_next are rewritten for the next item
        if (dynamic) {
            if (tid == 0)
                s_next = int64_t(atomicAdd(fp.counters, 1u));
            __syncthreads();
            it = s_next;
        } else {
            it += gridDim.x;
        }
    }

    if (dynamic && tid == 0) {
        // The last CTA to finish resets the counters for the next launch.
        __threadfence();
        const unsigned done = atomicAdd(fp.counters + 1, 1u);
        if (done == gridDim.x - 1) {
            atomicExch(fp.counters, 0u);
            atomicExch(fp.counters + 1, 0u);
        }
    }
}

using FoldKernel = void (*)(const FoldParams);

template <bool ACC>
FoldKernel pick_direct(int world)
{
    switch (world) {
    case 1: return fold_direct_kernel<1, 1, 4, ACC>;
    case 2: return fold_direct_kernel<2, 2, 4, ACC>;
    case 4: return fold_direct_kernel<4, 4, 4, ACC>;
    case 8: return fold_direct_kernel<8, 8, 2, ACC>;
    case 16: return fold_direct_kernel<16, 8, 2, ACC>;
    case 32: return fold_direct_kernel<32, 8, 2, ACC>;
    default: return fold_direct_kernel<0, 4, 2, ACC>;
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy kernel.  Warp 0 is the producer: one elected lane takes the work
// items (under the dynamic schedule it claims each from the device counter
// and posts its index through the item queue) and streams each item's W rank
// rows into a ring of shared-memory stages with cp.async.bulk (the TMA
// engine's non-tensor copy), one copy per rank per fill, completing on the
// stage's "full" mbarrier with a transaction count.
// Warps 1..4 consume a stage (fp32 adds in rank order from shared memory,
// scale, optional accumulate, 16-byte streaming stores) and release it on
// its "empty" mbarrier.  Every wait is bounded by %globaltimer: on expiry
// the kernel records a status word, stops issuing, waits (bounded) for the
// copies it already issued, and returns.

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `parity` to complete; false if `budget_ns` passed
// or another warp raised the abort flag first.
__device__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t budget_ns, volatile int32_t *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (abort_flag && *abort_flag)
            return false;
        if (global_ns() - t0 > budget_ns)
            return false;
    }
}

#ifndef TIDE_BULK_L2_EVICT_FIRST
#define TIDE_BULK_L2_EVICT_FIRST 0  // 1: bulk gradient loads carry an L2 evict-first policy (slower here)
#endif

// L2 policy for read-once gradient data (only used with TIDE_BULK_L2_EVICT_FIRST).
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
#if TIDE_BULK_L2_EVICT_FIRST
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy));
#else
    (void)policy;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)));
#endif
}

__device__ __forceinline__ uint4 lds_v4(const uint16_t *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

// Dynamic schedule of the bulk kernel: the producer lane claims work items
// from a device counter and hands them to the consumer warps through a queue
// of kItemQueue slots (item index, or -1 when the list is exhausted), each
// guarded by a "posted" and a "taken" mbarrier.
constexpr int kItemQueue = 8;

// Shared-memory layout of the bulk kernel: STAGES full + STAGES empty
// mbarriers, the abort flag, the item queue (posted and taken mbarriers,
// item slots), the producer's W source pointers, then the 128-byte aligned
// stage ring.
__host__ __device__ constexpr size_t bulk_ring_offset(int stages, int world)
{
    return ((size_t(2 * stages + 1 + 3 * kItemQueue) * 8 + size_t(world) * 8 + 127) / 128) * 128;
}

constexpr int kBulkMaxVec = 2;                               // vectors per consumer thread per chunk
constexpr int64_t kBulkMaxFill = 8 * kBulkMaxVec * 32 * kBulkConsumerWarps;  // 2048 elements
// Wide consumers (a CTA with the SM to itself): 4 vectors per thread, fills
// of up to 8,192 elements (16 KB of bf16) per rank, so that each bulk copy
// is larger (a copy costs a fixed ~60 ns per SM on top of its bytes).
constexpr int kWideVec = 4;
constexpr int64_t kBulkMaxFillWide = 8 * kWideVec * 32 * kBulkConsumerWarpsWide;  // 8192 elements

constexpr int32_t kStatusConsumerTimeout = 1;
constexpr int32_t kStatusProducerTimeout = 2;
constexpr int32_t kStatusDrainTimeout = 3;

// Summation orders (Section 4.3).  The W contributions to destination rank
// r are added in a sequence of positions q = 0..W-1; positions form groups
// of `group` consecutive entries whose partials are added in sequence order.
//   rank order:      q -> q, one group
//   one-node order:  every rank but r ascending, then r, one group
//   two-level order: node n = q / L: its ranks except n L + (r mod L)
//                    ascending, then that rank; groups of L (node partials)
__device__ __forceinline__ int seq_rank(int order, int q, int r, int W, int L)
{
    if (order == TIDE_ORDER_STAGED_OWN)
        return q == W - 1 ? r : (q < r ? q : q + 1);
    if (order == TIDE_ORDER_NODES) {
        const int n = q / L, l = q - n * L, own = r % L;
        return n * L + (l == L - 1 ? own : (l < own ? l : l + 1));
    }
    return q;
}

template <typename E>
__device__ __forceinline__ float ld_elem(const E *p);
template <>
__device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t *p)
{
    return ld_bf16(p);
}
template <>
__device__ __forceinline__ float ld_elem<float>(const float *p)
{
    return __ldg(p);
}

// Elements of a work item before its first 16-byte aligned source element,
// given the phase (elements past the last 16-byte boundary) that every
// rank's row shares at the item's start; at most `count`.
template <typename E>
__device__ __forceinline__ int64_t aligned_head(int32_t phase, int64_t count)
{
    constexpr int VE = 16 / int(sizeof(E));
    const int64_t h = (VE - phase) & (VE - 1);
    return h < count ? h : count;
}

// One element from global memory (pieces or tails the producer does not
// stage), in the plan's order.
template <bool ACC, typename E>
__device__ void fold_scalar_global(const uint64_t *bp, const FoldParams &fp, int r, int64_t src_off, float *dst)
{
    const int W = fp.world;
    float total = 0.0f;
    if (fp.order == TIDE_ORDER_TREE) {
        // Pairwise order as a binary counter: slot[l] holds the sum of a
        // complete subtree of 2^l ranks; rank q first absorbs the slots of
        // the set bits below q's lowest clear bit.  The slots left (the set
        // bits of W) are then added from the lowest level up.
        float slot[11];  // W <= 1024
        for (int q = 0; q < W; ++q) {
            float c = ld_elem<E>(reinterpret_cast<const E *>(bp[q]) + src_off);
            int l = 0;
            while ((q >> l) & 1) {
                c = __fadd_rn(slot[l], c);
                ++l;
            }
            slot[l] = c;
        }
        bool have = false;
        for (int l = 0; l < 11; ++l)
            if ((W >> l) & 1) {
                total = have ? __fadd_rn(slot[l], total) : slot[l];
                have = true;
            }
    } else {
        const int group = fp.order == TIDE_ORDER_NODES ? fp.node_size : W;
        float part = 0.0f;
        for (int q = 0; q < W; ++q) {
            const int u = seq_rank(fp.order, q, r, W, fp.node_size);
            const float x = ld_elem<E>(reinterpret_cast<const E *>(bp[u]) + src_off);
            const int l = q % group;
            part = l == 0 ? x : __fadd_rn(part, x);
            if (l == group - 1)
                total = q < group ? part : __fadd_rn(total, part);
        }
    }
    float y = __fmul_rn(fp.alpha, total);
    if (ACC)
        y = __fadd_rn(*dst, y);
    __stcs(dst, y);
}

// Eight consecutive elements of one rank from a shared-memory stage.
__device__ __forceinline__ void lds8(const uint16_t *p, float (&f)[8]) { unpack8(lds_v4(p), f); }
__device__ __forceinline__ void lds8(const float *p, float (&f)[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Tuning knob (compile-time, default on): add staged bf16 values into the
// fp32 sums with the mixed-precision add of sm_100 and later (widening is
// exact, the add rounds once to nearest even: the same result as widening
// first), one instruction per element instead of two.
#ifndef TIDE_BULK_MIXED_ADD
#define TIDE_BULK_MIXED_ADD 1
#endif

// acc[2i] += lo bf16 of w_i, acc[2i+1] += hi bf16 of w_i for the 4 words of x.
__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 &x)
{
#if TIDE_BULK_MIXED_ADD
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
            : "r"(w[i]));
#else
    float f[8];
    unpack8(x, f);
#pragma unroll
    for (int e = 0; e < 8; ++e)
        acc[e] = __fadd_rn(acc[e], f[e]);
#endif
}

template <typename E>
__device__ __forceinline__ void lds_add8(const E *p, float (&acc)[8]);
template <>
__device__ __forceinline__ void lds_add8<uint16_t>(const uint16_t *p, float (&acc)[8])
{
    add_bf16x8(acc, lds_v4(p));
}
template <>
__device__ __forceinline__ void lds_add8<float>(const float *p, float (&acc)[8])
{
    float f[8];
    lds8(p, f);
#pragma unroll
    for (int e = 0; e < 8; ++e)
        acc[e] = __fadd_rn(acc[e], f[e]);
}

__device__ __forceinline__ void add8(const float (&a)[8], float (&c)[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e)
        c[e] = __fadd_rn(a[e], c[e]);
}

__device__ __forceinline__ void copy8(const float (&a)[8], float (&c)[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e)
        c[e] = a[e];
}

// Tree order, one stage fill of nr <= 8 ranks (a power-of-two count, or the
// last fill): a binary counter over the fill's ranks with compile-time
// levels (slot[l]: complete subtree of 2^l ranks), then the slots of nr's
// set bits folded from the lowest level up into `part`, earlier ranks on
// the left of every addition.
template <typename E>
__device__ __forceinline__ void tree_fill(const E *sb, int64_t FILL, int64_t v, int nr, float (&part)[8])
{
    float s0[8], s1[8], s2[8], s3[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < nr) {
            float c[8];
            lds8(sb + size_t(j) * FILL + v * 8, c);
            if (j & 1) {
                add8(s0, c);
                if (j & 2) {
                    add8(s1, c);
                    if (j & 4) {
                        add8(s2, c);
                        copy8(c, s3);
                    } else {
                        copy8(c, s2);
                    }
                } else {
                    copy8(c, s1);
                }
            } else {
                copy8(c, s0);
            }
        }
    }
    bool have = false;
    if (nr & 1) {
        copy8(s0, part);
        have = true;
    }
    if (nr & 2) {
        if (have) add8(s1, part); else copy8(s1, part);
        have = true;
    }
    if (nr & 4) {
        if (have) add8(s2, part); else copy8(s2, part);
        have = true;
    }
    if (nr & 8) {
        if (have) add8(s3, part); else copy8(s3, part);
    }
}

// Tree order, a full fill of N = 2^k ranks: the balanced tree with
// compile-time shape, e.g. ((x0+x1)+(x2+x3))+((x4+x5)+(x6+x7)) for N = 8.
template <int N, typename E>
__device__ __forceinline__ void tree_fill_pow2(const E *sb, int64_t FILL, int64_t v, float (&part)[8])
{
    float x[N][8];
#pragma unroll
    for (int j = 0; j < N; ++j)
        lds8(sb + size_t(j) * FILL + v * 8, x[j]);
    // After the level of width h, the subtree of ranks [j, j + 2h) is held in
    // x[j + 2h - 1]; its left half (the earlier ranks) in x[j + h - 1].
#pragma unroll
    for (int h = 1; h < N; h *= 2)
#pragma unroll
        for (int j = 0; j < N; j += 2 * h)
            add8(x[j + h - 1], x[j + 2 * h - 1]);
    copy8(x[N - 1], part);
}

// Tree order across fills: push the partial of complete fill g into the
// counter x (x[l]: complete subtree of 2^l fills; g < 2^LV - 1).  g is the
// same for the whole CTA, so the switch is a uniform branch and every slot
// index is a compile-time constant.
template <int LV>
__device__ __forceinline__ void tree_push(float (&x)[LV][8], int g, float (&part)[8])
{
    const int t = __ffs(~g) - 1;  // trailing ones of g: the slots this fill absorbs
#pragma unroll
    for (int l = 0; l < LV; ++l) {
        if (l == t) {
#pragma unroll
            for (int m = 0; m < l; ++m)
                add8(x[m], part);
            copy8(part, x[l]);
        }
    }
}

// Consumer modes of the bulk kernel: one chain in the sequence the producer
// stages (rank and one-node orders), node partials (two-level order), or the
// pairwise tree: all ranks in one fill (no counter), up to 2^3 - 1 full fills
// per chunk, or up to 2^kTreeLevels - 1 (each counter level costs 8
// registers per vector, so the smaller counters keep two vectors per thread).
enum { kModeChain = 0, kModeNodes = 1, kModeTreeOne = 2, kModeTree = 3, kModeTreeDeep = 4 };
constexpr int kTreeLevelsShallow = 3;

template <int MODE>
struct TreeShape {
    static constexpr bool tree = MODE >= kModeTreeOne;
    static constexpr int levels = MODE == kModeTreeDeep ? kTreeLevels : MODE == kModeTree ? kTreeLevelsShallow : 0;
    static constexpr int vec = MODE == kModeTreeDeep ? 1 : kBulkMaxVec;  // vectors per consumer thread
};

// ACC: accumulate into the existing shard.  E: gradient element (uint16_t =
// bf16, float = fp32).  MODE: how the consumers combine the staged ranks.
// CW: consumer warps (4, two CTAs per SM; or 8, one vector each, for a CTA
// that has the SM to itself).
template <bool ACC, typename E, int MODE, int CW = kBulkConsumerWarps>
__global__ void __launch_bounds__(32 * (1 + CW), CW == kBulkConsumerWarps ? 2 : 1)
    fold_bulk_kernel(const FoldParams fp)
{
    constexpr bool GROUPED = MODE == kModeNodes;
    constexpr bool TREE = TreeShape<MODE>::tree;
    constexpr int LV = TreeShape<MODE>::levels;
    constexpr int NV = TREE ? TreeShape<MODE>::vec : CW == kBulkConsumerWarps ? kBulkMaxVec : kWideVec;
    extern __shared__ __align__(128) unsigned char smem[];
    const int W = fp.world;
    const int RG = fp.fill_ranks;          // ranks per stage fill
    const int NG = (W + RG - 1) / RG;      // fills per chunk of FILL elements
    const int STAGES = fp.stages;
    const int64_t FILL = fp.fill_elems;
    const int L = GROUPED ? fp.node_size : W;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(empty + STAGES);
    uint64_t *q_posted = empty + STAGES + 1;
    uint64_t *q_taken = q_posted + kItemQueue;
    volatile int64_t *q_item = reinterpret_cast<volatile int64_t *>(q_taken + kItemQueue);
    const E **src_cache = reinterpret_cast<const E **>(q_taken + 2 * kItemQueue);  // producer's W pointers, in order
    E *ring = reinterpret_cast<E *>(smem + bulk_ring_offset(STAGES, W));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float alpha = fp.alpha;
    const bool dyn = fp.sched == TIDE_SCHED_DYNAMIC;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        for (int s = 0; s < kItemQueue; ++s) {
            mbar_init(&q_posted[s], 1);
            mbar_init(&q_taken[s], CW);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        if (lane != 0)
            return;
        // ------------------------------------------------------------ producer
        // For every chunk of FILL elements of a work item, NG stage fills of
        // RG ranks each, in the plan's summation sequence.
        uint32_t stage = 0, phase = 0;
        int64_t fills = 0, skipped = -1;
        bool stop = false;
        const uint64_t policy = TIDE_BULK_L2_EVICT_FIRST ? evict_first_policy() : 0;
        uint32_t qk = 0;  // item-queue position (dynamic schedule)
        for (int64_t it = blockIdx.x; !stop; it += gridDim.x) {
            if (dyn) {
                // claim the next item and post it (or -1) to the consumers
                const uint32_t qs = qk % kItemQueue, qpar = (qk / kItemQueue) & 1u;
                if (!mbar_wait_bounded(&q_taken[qs], qpar ^ 1u, fp.wait_budget_ns, abort_flag)) {
                    if (!*abort_flag)
                        atomicExch(fp.status, kStatusProducerTimeout);
                    *abort_flag = 1;
                    break;
                }
                const int64_t t = int64_t(atomicAdd(fp.counters, 1u));
                it = t < fp.n_items ? t : -1;
                q_item[qs] = it;
                mbar_arrive(&q_posted[qs]);
                ++qk;
                if (it < 0)
                    break;
            } else if (it >= fp.n_items) {
                break;
            }
            const Item item = fp.items[it];
            const Seg seg = fp.segs[item.seg];
            if ((item.count_kind & kItemPad) || seg.src_phase < 0)
                continue;
            const int64_t total = int64_t(item.count_kind & ~kItemPad);
            const int64_t head = aligned_head<E>(seg.src_phase, total);  // the consumers fold these directly
            const int64_t count = total - head;
            const uint64_t *bp = fp.ptrs + int64_t(seg.param) * W;
            const int64_t base = seg.src_elem + item.begin + head;
            for (int q = 0; q < W; ++q)
                src_cache[q] = reinterpret_cast<const E *>(bp[seq_rank(fp.order, q, seg.rank, W, fp.node_size)]) + base;
            for (int64_t c = 0; c < count && !stop; c += FILL) {
                const int64_t len = count - c < FILL ? count - c : FILL;
                const uint32_t bytes = uint32_t(len & ~int64_t(7)) * uint32_t(sizeof(E));
                for (int g = 0; g < NG; ++g) {
                    const int u0 = g * RG;
                    const int nr = W - u0 < RG ? W - u0 : RG;
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, fp.wait_budget_ns, abort_flag)) {
                        if (!*abort_flag)
                            atomicExch(fp.status, kStatusProducerTimeout);
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                    if ((fp.debug & TIDE_DEBUG_SKIP_FILL) && it == 0 && c == 0 && g == 0) {
                        skipped = fills;  // leave work item 0's first stage unfilled: its consumers' wait expires
                    } else {
                        mbar_arrive_expect_tx(&full[stage], uint32_t(nr) * bytes);
                        if (bytes) {
                            E *dst = ring + size_t(stage) * RG * FILL;
#pragma unroll 4
                            for (int j = 0; j < nr; ++j)
                                bulk_copy_g2s(dst + size_t(j) * FILL, src_cache[u0 + j] + c, bytes, &full[stage], policy);
                        }
                    }
                    ++fills;
                    if (++stage == uint32_t(STAGES)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        // Drain: the last fills of each stage must land before this CTA exits.
        const int64_t first = fills > STAGES ? fills - STAGES : 0;
        for (int64_t f = first; f < fills; ++f) {
            if (f == skipped)
                continue;
            const uint32_t s = uint32_t(f % STAGES), par = uint32_t((f / STAGES) & 1);
            if (!mbar_wait_bounded(&full[s], par, fp.wait_budget_ns, nullptr))
                atomicExch(fp.status, kStatusDrainTimeout);
        }
        if (dyn) {
            // The last CTA to finish claiming resets the counters for the
            // next launch (every producer lane gets here, even after a timeout).
            __threadfence();
            const unsigned done = atomicAdd(fp.counters + 1, 1u);
            if (done == gridDim.x - 1) {
                atomicExch(fp.counters, 0u);
                atomicExch(fp.counters + 1, 0u);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Each consumer thread owns up to NV 8-element vectors of a
    // chunk and keeps their fp32 sums in registers across the chunk's NG
    // fills, so the contributions are added in the plan's sequence.
    const int ctid = threadIdx.x - 32;
    constexpr int NCT = 32 * CW;
    uint32_t stage = 0, phase = 0;
    uint32_t qk = 0;  // item-queue position (dynamic schedule)
    for (int64_t it = blockIdx.x;; it += gridDim.x) {
        if (dyn) {
            const uint32_t qs = qk % kItemQueue, qpar = (qk / kItemQueue) & 1u;
            if (!mbar_wait_bounded(&q_posted[qs], qpar, fp.wait_budget_ns, abort_flag)) {
                if (!*abort_flag)
                    atomicExch(fp.status, kStatusConsumerTimeout);
                *abort_flag = 1;
                return;
            }
            it = q_item[qs];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&q_taken[qs]);
            ++qk;
            if (it < 0)
                break;
        } else if (it >= fp.n_items) {
            break;
        }
        const Item item = fp.items[it];
        const Seg seg = fp.segs[item.seg];
        const int64_t total = int64_t(item.count_kind & ~kItemPad);
        const bool pad = (item.count_kind & kItemPad) != 0;
        float *dst0 = fp.out + int64_t(seg.rank) * fp.stride + seg.dst_elem + (pad ? seg.n_valid : 0) + item.begin;
        const uint64_t *bp = fp.ptrs + int64_t(seg.param) * W;
        if (pad) {
            const float y = __fmul_rn(alpha, 0.0f);
            for (int64_t e = ctid; e < total; e += NCT)
                __stcs(dst0 + e, ACC ? __fadd_rn(dst0[e], y) : y);
            continue;
        }
        if (seg.src_phase < 0) {  // the ranks' rows differ in 16-byte phase: no bulk copies
            for (int64_t e = ctid; e < total; e += NCT)
                fold_scalar_global<ACC, E>(bp, fp, seg.rank, seg.src_elem + item.begin + e, dst0 + e);
            continue;
        }
        // Every rank's row shares one phase: the elements before the first
        // 16-byte boundary are folded from global memory, the rest is staged.
        const int64_t head = aligned_head<E>(seg.src_phase, total);
        for (int64_t e = ctid; e < head; e += NCT)
            fold_scalar_global<ACC, E>(bp, fp, seg.rank, seg.src_elem + item.begin + e, dst0 + e);
        const int64_t count = total - head;
        const int64_t src_at = seg.src_elem + item.begin + head;
        float *dst = dst0 + head;
        const bool dst_vec = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
        for (int64_t c = 0; c < count; c += FILL) {
            const int64_t len = count - c < FILL ? count - c : FILL;
            const int64_t nv = len >> 3;
            float acc[NV][8];
            float part[GROUPED ? NV : 1][8];
            float tx[TREE ? NV : 1][LV > 0 ? LV : 1][8];
            float old[NV][8];
            if (ACC) {
                // Issue the loads of the existing shard values before waiting
                // for the chunk's fills, so their latency overlaps the copies.
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t v = ctid + int64_t(k) * NCT;
                    if (v < nv)
                        load8(dst + c + v * 8, old[k], dst_vec);
                }
            }
            for (int g = 0; g < NG; ++g) {
                const int u0 = g * RG;
                const int nr = W - u0 < RG ? W - u0 : RG;
                if (!mbar_wait_bounded(&full[stage], phase, fp.wait_budget_ns, abort_flag)) {
                    if (!*abort_flag)
                        atomicExch(fp.status, kStatusConsumerTimeout);
                    *abort_flag = 1;
                    return;
                }
                const E *sb = ring + size_t(stage) * RG * FILL;
                if constexpr (GROUPED) {
                    // The fill's ranks, as runs of consecutive ranks of one
                    // node; the runs are the same for every vector, so they
                    // are walked once, each run over all of this thread's
                    // vectors.  After the first run, runs start on a node.
                    int l = u0 % L;
                    for (int j = 0; j < nr;) {
                        const int run = nr - j < L - l ? nr - j : L - l;
                        const bool node_end = l + run == L, first_node = u0 + j < L;
#pragma unroll
                        for (int k = 0; k < NV; ++k) {
                            const int64_t v = ctid + int64_t(k) * NCT;
                            if (v < nv) {
                                const E *p0 = sb + size_t(j) * FILL + v * 8;
                                if (l == 0)
                                    lds8(p0, part[k]);
                                else
                                    lds_add8(p0, part[k]);
#pragma unroll 4
                                for (int t = 1; t < run; ++t)
                                    lds_add8(p0 + size_t(t) * FILL, part[k]);
                                if (node_end) {  // node complete: add its partial
                                    if (first_node) {
                                        copy8(part[k], acc[k]);
                                    } else {
#pragma unroll
                                        for (int e = 0; e < 8; ++e)
                                            acc[k][e] = __fadd_rn(acc[k][e], part[k][e]);
                                    }
                                }
                            }
                        }
                        j += run;
                        l = 0;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        const int64_t v = ctid + int64_t(k) * NCT;
                        if (v < nv) {
                            if constexpr (TREE) {
                                float p[8];
                                if (nr == 8)
                                    tree_fill_pow2<8>(sb, FILL, v, p);
                                else if (nr == 4)
                                    tree_fill_pow2<4>(sb, FILL, v, p);
                                else if (nr == 2)
                                    tree_fill_pow2<2>(sb, FILL, v, p);
                                else
                                    tree_fill(sb, FILL, v, nr, p);
                                if constexpr (LV == 0)
                                    copy8(p, acc[k]);  // the one fill holds every rank
                                else if (nr == RG)
                                    tree_push<LV>(tx[k], g, p);
                                else
                                    copy8(p, acc[k]);  // the last fill, short: its partial waits in acc
                            } else {
                                int j0 = 0;
                                if (g == 0) {
                                    lds8(sb + v * 8, acc[k]);
                                    j0 = 1;
                                }
#pragma unroll 4
                                for (int j = j0; j < nr; ++j)
                                    lds_add8(sb + size_t(j) * FILL + v * 8, acc[k]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[stage]);
                if (++stage == uint32_t(STAGES)) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if constexpr (TREE && LV > 0) {
                // The counter's slots (set bits of the full-fill count) join
                // the short fill's partial from the lowest level up.
                const int nfull = W / RG;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    bool have = nfull * RG != W;
#pragma unroll
                    for (int l = 0; l < LV; ++l) {
                        if ((nfull >> l) & 1) {
                            if (have) add8(tx[k][l], acc[k]); else copy8(tx[k][l], acc[k]);
                            have = true;
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int64_t v = ctid + int64_t(k) * NCT;
                if (v < nv)
                    store8_onto<ACC>(dst + c + v * 8, acc[k], old[k], alpha, dst_vec);
            }
            for (int64_t e = nv * 8 + ctid; e < len; e += NCT)
                fold_scalar_global<ACC, E>(bp, fp, seg.rank, src_at + c + e, dst + c + e);
        }
    }
}

template <bool ACC, typename E>
FoldKernel pick_bulk_mode(int order, int fills, int full_fills)
{
    if (order == TIDE_ORDER_NODES)
        return fold_bulk_kernel<ACC, E, kModeNodes>;
    if (order == TIDE_ORDER_TREE) {
        if (fills == 1)
            return fold_bulk_kernel<ACC, E, kModeTreeOne>;
        if (full_fills < (1 << kTreeLevelsShallow))
            return fold_bulk_kernel<ACC, E, kModeTree>;
        return fold_bulk_kernel<ACC, E, kModeTreeDeep>;
    }
    return fold_bulk_kernel<ACC, E, kModeChain>;
}

// The tree counter's depth follows the stage fills per chunk: `fills` in
// all, `full_fills` of them holding fill_ranks ranks.  `cw`: consumer warps
// (bulk_consumer_warps; the tree order has no wide form).
template <bool ACC>
FoldKernel pick_bulk(int dtype, int order, int world, int fill_ranks, int cw = kBulkConsumerWarps)
{
    constexpr int CW = kBulkConsumerWarpsWide;
    if (cw == CW && order == TIDE_ORDER_NODES)
        return dtype == TIDE_DTYPE_F32 ? fold_bulk_kernel<ACC, float, kModeNodes, CW>
                                       : fold_bulk_kernel<ACC, uint16_t, kModeNodes, CW>;
    if (cw == CW && (order == TIDE_ORDER_RANK_ASC || order == TIDE_ORDER_STAGED_OWN))
        return dtype == TIDE_DTYPE_F32 ? fold_bulk_kernel<ACC, float, kModeChain, CW>
                                       : fold_bulk_kernel<ACC, uint16_t, kModeChain, CW>;
    const int fills = (world + fill_ranks - 1) / fill_ranks, full_fills = world / fill_ranks;
    return dtype == TIDE_DTYPE_F32 ? pick_bulk_mode<ACC, float>(order, fills, full_fills)
                                   : pick_bulk_mode<ACC, uint16_t>(order, fills, full_fills);
}

}  // namespace

BulkShape bulk_shape(int world, int64_t fill_elems, int fill_ranks, bool whole_sm, int elem_bytes, int order)
{
    // Default: 4 KB of each of up to 8 ranks per stage fill (32 KB stages),
    // three stages per CTA, two CTAs per SM.  Wider groups take several fills
    // per chunk; the consumers keep the partial sums in registers meanwhile.
    // The tree order: fills of a power-of-two number of ranks (at most 8), so
    // that every full fill is a complete subtree; with 8 or more full fills
    // per chunk (the deep counter) one vector per consumer thread, so half
    // the fill.
    // A CTA with the SM to itself and wide consumers: 16 KB per rank per
    // copy, 4 ranks per fill (64 KB stages, three in the ring): at small CTA
    // budgets each SM is limited by its per-copy cost, not HBM.
    const bool tree = order == TIDE_ORDER_TREE;
    const bool wide_sm = bulk_consumer_warps(whole_sm, order, elem_bytes == 4 ? TIDE_DTYPE_F32 : TIDE_DTYPE_BF16) ==
                         kBulkConsumerWarpsWide;
    BulkShape b{};
    int rg = fill_ranks > 0 ? fill_ranks : wide_sm ? 4 : 8;
    if (tree && rg > 8)
        rg = 8;
    if (rg >= world)
        rg = world;
    else if (tree)
        while (rg & (rg - 1))
            rg &= rg - 1;  // largest power of two not above it
    const bool deep = tree && rg < world && world / rg >= (1 << kTreeLevelsShallow);
    const int64_t max_fill = deep ? kBulkMaxFill / kBulkMaxVec : wide_sm ? kBulkMaxFillWide : kBulkMaxFill;
    int64_t fill = fill_elems > 0 ? fill_elems : wide_sm ? 16384 / elem_bytes : 4096 / elem_bytes;
    if (fill > max_fill)
        fill = max_fill;
    fill &= ~int64_t(7);
    if (fill < 8)
        fill = 8;
    while (fill > 8 && fill * rg * elem_bytes * 2 > 200 * 1024)  // two stages must fit in shared memory
        fill = (fill / 2) & ~int64_t(7);
    const int64_t stage_bytes = fill * rg * elem_bytes;
    // A CTA that has an SM to itself (small CTA budgets) takes twice the ring.
    int64_t stages = (whole_sm ? 2 * kBulkSmemTarget : kBulkSmemTarget) / stage_bytes;
    if (stages > 16)
        stages = 16;
    if (stages < 2)
        stages = 2;
    b.fill_elems = int32_t(fill);
    b.fill_ranks = rg;
    b.stages = int32_t(stages);
    b.smem_bytes = bulk_ring_offset(int(stages), world) + size_t(stages * stage_bytes);
    return b;
}

size_t fold_smem_bytes(int kernel, int world, int64_t fill_elems, int fill_ranks, bool whole_sm, int elem_bytes,
                       int order)
{
    if (kernel == TIDE_KERNEL_BULK)
        return bulk_shape(world, fill_elems, fill_ranks, whole_sm, elem_bytes, order).smem_bytes;
    return size_t(world) * sizeof(uint64_t);
}

cudaError_t fold_occupancy(int kernel, int world, int block, size_t smem, int *blocks_per_sm, int dtype, int order,
                           int fill_ranks, int consumer_warps)
{
    if (kernel == TIDE_KERNEL_BULK) {
        // Allow the device maximum once per kernel instance: it serves every
        // world size and stage shape.
        int dev = 0, optin = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess)
            return e;
        if (smem > size_t(optin))
            return cudaErrorInvalidValue;
        const int rg = bulk_shape(world, 0, fill_ranks, false, dtype == TIDE_DTYPE_F32 ? 4 : 2, order).fill_ranks;
        const int cw = consumer_warps;
        for (int acc = 0; acc < 2; ++acc) {
            FoldKernel k = acc ? pick_bulk<true>(dtype, order, world, rg, cw)
                               : pick_bulk<false>(dtype, order, world, rg, cw);
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
            if (e != cudaSuccess)
                return e;
        }
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            blocks_per_sm, pick_bulk<false>(dtype, order, world, rg, cw), block, smem);
    }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, pick_direct<false>(world), block, smem);
}

cudaError_t launch_fold(const FoldParams &fp, int kernel, int accumulate, int grid, int block, size_t smem,
                        cudaStream_t stream)
{
    FoldKernel k;
    if (kernel == TIDE_KERNEL_BULK)
        k = accumulate ? pick_bulk<true>(fp.dtype, fp.order, fp.world, fp.fill_ranks, fp.consumer_warps)
                       : pick_bulk<false>(fp.dtype, fp.order, fp.world, fp.fill_ranks, fp.consumer_warps);
    else
        k = accumulate ? pick_direct<true>(fp.world) : pick_direct<false>(fp.world);
    k<<<grid, block, smem, stream>>>(fp);
    return cudaGetLastError();
}

}  // namespace tide

// All-gather placement kernel: TIDE paper Section 2.1, Equation (2).  Rank r's
// shard of parameter p sits in the rank-major input at slot r, offset o_p; its
// v_{p,r} real rows land at rows [r R_p, r R_p + v_{p,r}) of the full tensor,
// which is the contiguous element range starting at r R_p K_p.  Padding rows
// are never read.  A pure HBM copy: one short CTA per (piece, chunk) work
// item moves 16-byte vectors.  When source and destination differ in 16-byte
// phase, each aligned 16-byte store is assembled from the two aligned source
// vectors that cover its eight elements (a shift by the phase difference).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tide_internal.h"

namespace tide {
namespace {

__device__ __forceinline__ uint4 ld_once_v4(const uint16_t *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

constexpr int kAgUnroll = 8;  // 16-byte vectors in flight per thread: enough to cover HBM latency

// Eight bf16 values starting `sh` (1..7) halfwords into the 32 bytes a, b
// (two consecutive aligned source vectors): output word m is the 32 bits
// starting sh halfwords past word m of the pair.  sh is uniform across the
// CTA, so the switch does not diverge and every word index is a constant.
__device__ __forceinline__ uint4 shift_halfwords(const uint4 &a, const uint4 &b, int sh)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
    switch (sh) {
#define TIDE_SHIFT_CASE(S)                                                                     \
    case S:                                                                                    \
        _Pragma("unroll") for (int m = 0; m < 4; ++m) o[m] =                                   \
            (S & 1) ? __byte_perm(w[S / 2 + m], w[S / 2 + m + 1], 0x5432) : w[S / 2 + m];      \
        break;
        TIDE_SHIFT_CASE(1)
        TIDE_SHIFT_CASE(2)
        TIDE_SHIFT_CASE(3)
        TIDE_SHIFT_CASE(4)
        TIDE_SHIFT_CASE(5)
        TIDE_SHIFT_CASE(6)
        default:
        TIDE_SHIFT_CASE(7)
#undef TIDE_SHIFT_CASE
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Copy `count` bf16 elements when source and destination differ in 16-byte
// phase.  After the destination's head, destination vector v takes source
// elements [8v, 8v + 8) past the head, which straddle the aligned source
// vectors a_v and a_{v+1}; both are loaded (each aligned 16-byte load holds at
// least one element of the range, so it stays inside the source's pages) and
// shifted into place.  Heads and tails: batched scalar loads, then stores.
template <int NT>
__device__ __forceinline__ void place_shifted(const uint16_t *src, uint16_t *dst, int64_t count, int tid)
{
    const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
    int64_t h = int64_t(((16u - (da & 15u)) & 15u) >> 1);
    if (h > count)
        h = count;
    const int64_t nv = (count - h) >> 3;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src + h);
    const uint16_t *sa = reinterpret_cast<const uint16_t *>(s0 & ~uintptr_t(15));
    const int sh = int((s0 & 15u) >> 1);  // nonzero: the phases differ
    uint4 *d8 = reinterpret_cast<uint4 *>(dst + h);
    constexpr int U = 1;  // one pair of source vectors per thread per pass: keeps the kernel at 4 CTAs per SM
    for (int64_t v = tid; v < nv; v += int64_t(NT) * U) {
        uint4 a[U], b[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t vj = v + int64_t(j) * NT;
            if (vj < nv) {
                a[j] = ld_once_v4(sa + vj * 8);
                b[j] = ld_once_v4(sa + vj * 8 + 8);
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t vj = v + int64_t(j) * NT;
            if (vj < nv)
                d8[vj] = shift_halfwords(a[j], b[j], sh);
        }
    }
    // head [0, h) and tail [h + 8 nv, count): at most 14 elements
    const int64_t e = tid < h ? tid : h + nv * 8 + (tid - h);
    if (tid < 16 && e < count)
        dst[e] = src[e];
}

template <int NP>
__global__ void __launch_bounds__(kAgThreads) ag_place_kernel(const __grid_constant__ AgParamsT<NP> ap)
{
    constexpr int NT = kAgThreads;
    const int tid = threadIdx.x;
    for (int64_t i = ap.item_begin + blockIdx.x; i < ap.item_end; i += gridDim.x) {
        const Item item = ap.items[i];
        const Seg seg = ap.segs[item.seg];
        const int64_t count = int64_t(item.count_kind & ~kItemPad);
        const uint16_t *src = ap.slots + int64_t(seg.rank) * ap.stride + seg.dst_elem + item.begin;
        uint16_t *dst = ap.full[seg.param - ap.param_base] + seg.src_elem + item.begin;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
        if (((sa ^ da) & 15u) == 0) {
            int64_t h = int64_t(((16u - (sa & 15u)) & 15u) >> 1);
            if (h > count)
                h = count;
            const int64_t nv = (count - h) >> 3;
            const uint16_t *s8 = src + h;
            uint4 *d8 = reinterpret_cast<uint4 *>(dst + h);
            for (int64_t v = tid; v < nv; v += int64_t(NT) * kAgUnroll) {
                uint4 x[kAgUnroll];
#pragma unroll
                for (int j = 0; j < kAgUnroll; ++j) {
                    const int64_t vj = v + int64_t(j) * NT;
                    if (vj < nv)
                        x[j] = ld_once_v4(s8 + vj * 8);
                }
#pragma unroll
                for (int j = 0; j < kAgUnroll; ++j) {
                    const int64_t vj = v + int64_t(j) * NT;
                    if (vj < nv)
                        d8[vj] = x[j];
                }
            }
            for (int64_t e = tid; e < h; e += NT)
                dst[e] = src[e];
            for (int64_t e = h + nv * 8 + tid; e < count; e += NT)
                dst[e] = src[e];
        } else {
            place_shifted<NT>(src, dst, count, tid);
        }
    }
}

// Two fp32 values rounded to nearest even and packed as a bf16 pair (low half first).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Mixed-precision placement (fp32 master shards -> bf16 full tensors): the
// same walk as ag_place_kernel, reading 32 bytes of fp32 and writing 16 bytes
// of bf16 per vector when, after a common head, both sides are 16-byte aligned.
template <int NP>
__global__ void __launch_bounds__(kAgThreads) ag_cast_kernel(const __grid_constant__ AgParamsT<NP> ap)
{
    constexpr int NT = kAgThreads;
    constexpr int U = 4;  // 8-element vectors in flight per thread
    const int tid = threadIdx.x;
    for (int64_t i = ap.item_begin + blockIdx.x; i < ap.item_end; i += gridDim.x) {
        const Item item = ap.items[i];
        const Seg seg = ap.segs[item.seg];
        const int64_t count = int64_t(item.count_kind & ~kItemPad);
        const float *src = ap.slots_f32 + int64_t(seg.rank) * ap.stride + seg.dst_elem + item.begin;
        uint16_t *dst = ap.full[seg.param - ap.param_base] + seg.src_elem + item.begin;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
        int64_t h = int64_t(((16u - (da & 15u)) & 15u) >> 1);
        if (h > count)
            h = count;
        if (((sa + uintptr_t(h) * 4u) & 15u) == 0) {
            const int64_t nv = (count - h) >> 3;
            const float4 *s4 = reinterpret_cast<const float4 *>(src + h);
            uint4 *d8 = reinterpret_cast<uint4 *>(dst + h);
            for (int64_t v = tid; v < nv; v += int64_t(NT) * U) {
                float4 a[U], b[U];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const int64_t vj = v + int64_t(j) * NT;
                    if (vj < nv) {
                        a[j] = __ldcs(s4 + 2 * vj);
                        b[j] = __ldcs(s4 + 2 * vj + 1);
                    }
                }
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const int64_t vj = v + int64_t(j) * NT;
                    if (vj < nv)
                        d8[vj] = make_uint4(pack_bf16x2(a[j].x, a[j].y), pack_bf16x2(a[j].z, a[j].w),
                                            pack_bf16x2(b[j].x, b[j].y), pack_bf16x2(b[j].z, b[j].w));
                }
            }
            for (int64_t e = tid; e < h; e += NT)
                dst[e] = to_bf16_bits(src[e]);
            for (int64_t e = h + nv * 8 + tid; e < count; e += NT)
                dst[e] = to_bf16_bits(src[e]);
        } else {
            // Phases differ: coalesced scalar loads, eight in flight per
            // thread before their stores.
            constexpr int B = 2;
            for (int64_t e = tid; e < count; e += int64_t(NT) * B) {
                float x[B];
#pragma unroll
                for (int j = 0; j < B; ++j) {
                    const int64_t ej = e + int64_t(j) * NT;
                    if (ej < count)
                        x[j] = __ldcs(src + ej);
                }
#pragma unroll
                for (int j = 0; j < B; ++j) {
                    const int64_t ej = e + int64_t(j) * NT;
                    if (ej < count)
                        dst[ej] = to_bf16_bits(x[j]);
                }
            }
        }
    }
}

}  // namespace

// Tuning knob (compile-time; default: leave the driver's choice): the
// placements' preferred shared-memory carveout, in percent.  The fold runs
// with two 98 KB rings per SM; a placement that asks for the same carveout
// lets the SMs switch between the two kernels without reconfiguring.
#ifndef TIDE_AG_CARVEOUT
#define TIDE_AG_CARVEOUT -1
#endif

namespace {
template <typename K>
cudaError_t prefer_carveout(K kernel)
{
    if (TIDE_AG_CARVEOUT < 0)
        return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, TIDE_AG_CARVEOUT);
}

AgParamsT<kAgParamsSmall> small_params(const AgParams &ap)
{
    AgParamsT<kAgParamsSmall> s;
    s.segs = ap.segs;
    s.items = ap.items;
    s.item_begin = ap.item_begin;
    s.item_end = ap.item_end;
    s.slots = ap.slots;
    s.slots_f32 = ap.slots_f32;
    s.stride = ap.stride;
    s.param_base = ap.param_base;
    s.n_full = ap.n_full;
    for (int i = 0; i < kAgParamsSmall; ++i)
        s.full[i] = i < ap.n_full ? ap.full[i] : nullptr;
    return s;
}
}  // namespace

cudaError_t launch_ag(const AgParams &ap, int grid, cudaStream_t stream)
{
    if (ap.n_full <= kAgParamsSmall) {
        static const cudaError_t carve = prefer_carveout(ag_place_kernel<kAgParamsSmall>);
        if (carve != cudaSuccess)
            return carve;
        ag_place_kernel<kAgParamsSmall><<<grid, kAgThreads, 0, stream>>>(small_params(ap));
    } else {
        static const cudaError_t carve = prefer_carveout(ag_place_kernel<kAgParamsPerLaunch>);
        if (carve != cudaSuccess)
            return carve;
        ag_place_kernel<kAgParamsPerLaunch><<<grid, kAgThreads, 0, stream>>>(ap);
    }
    return cudaGetLastError();
}

cudaError_t launch_ag_f32(const AgParams &ap, int grid, cudaStream_t stream)
{
    if (ap.n_full <= kAgParamsSmall) {
        static const cudaError_t carve = prefer_carveout(ag_cast_kernel<kAgParamsSmall>);
        if (carve != cudaSuccess)
            return carve;
        ag_cast_kernel<kAgParamsSmall><<<grid, kAgThreads, 0, stream>>>(small_params(ap));
    } else {
        static const cudaError_t carve = prefer_carveout(ag_cast_kernel<kAgParamsPerLaunch>);
        if (carve != cudaSuccess)
            return carve;
        ag_cast_kernel<kAgParamsPerLaunch><<<grid, kAgThreads, 0, stream>>>(ap);
    }
    return cudaGetLastError();
}

}  // namespace tide

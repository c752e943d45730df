/*
 * tide.h -- C ABI of the GB300 layout-folded reduce-scatter (TIDE-RS fold)
 * and all-gather placement (TIDE-AG addressing) for FSDP2 parameter groups.
 *
 * Source of the operations: "The Endgame of FSDP Communication: Layout-Aware
 * Collectives on Copy Engines, RDMA, and NVSwitch" (TIDE).
 *   - Section 2.1 and Table 2: dim-0 shard geometry.  Parameter p is viewed as
 *     (D_p, K_p); each of the W ranks owns R_p = ceil(D_p / W) rows (rows past
 *     D_p are zero padding); rank shards are concatenated parameter-major at
 *     prefix offsets o_p inside one rank slot of S = sum_p R_p K_p elements.
 *   - Section 4, Equation (5): out_{p,r} <- (accumulate ? out_{p,r} : 0)
 *       + alpha * sum_{u=0}^{W-1} G_p^(u)[rows of rank r].
 *   - Section 2.1, Equation (2): all-gather landing; rank r's shard of p moves
 *     from slot r, offset o_p to rows [r R_p, r R_p + v_{p,r}) of the full
 *     parameter tensor, padding dropped.
 *   - Section 6: no metadata is copied to the GPU per call; the gradient
 *     pointer table is uploaded once when the plan is built (or rebound).
 *
 * Here all W ranks are virtual: their gradients and shard slots are W sets
 * of buffers in the same GPU's memory, and the collective becomes one W-way
 * gather-sum kernel (reduce-scatter) and one placement kernel or copy-engine
 * copy (all-gather).  There is no inter-GPU traffic.
 *
 * Conventions for every call:
 *   - Ownership: the caller owns every tensor (gradients, fp32 shards, bf16
 *     slots, full parameters).  A plan owns only its device tables and the
 *     streams and events of its copy-engine placement (created in
 *     tide_plan_build, released in tide_plan_destroy).  tide_rs_fold and the
 *     placements allocate no device memory.
 *   - Pointers named "device" must be CUDA device (or managed) memory of the
 *     current device; pointers named "host" are ordinary host memory read
 *     before the call returns.
 *   - Streams are cudaStream_t values passed as void*; NULL is the legacy
 *     default stream.  Hot calls are asynchronous and stream-ordered; a plan
 *     must not be used on two streams at once without caller synchronisation.
 *     tide_rs_fold, tide_ag_place (every mode) and tide_ag_place_f32 may be
 *     captured into a CUDA graph; in the copy-engine modes the capture takes
 *     in the plan's internal streams (forked from and joined back to the
 *     capturing stream), and a replay issues the whole copy list at once.
 *     The graph reads the plan's tables, so the plan must outlive every
 *     replay (tide_plan_destroy of a plan that was captured synchronises the
 *     device before freeing).
 *   - Errors are returned as tide_status_t, never thrown; on failure nothing
 *     was enqueued.  tide_last_error() gives a human-readable detail for the
 *     last failing call on the calling thread.
 *   - Numerics: bf16 -> fp32 widening is exact; the W contributions are added
 *     in fp32, round-to-nearest-even, in the plan's order -- by default rank
 *     order 0, 1, ..., W-1 starting from rank 0's value; then y = alpha * sum;
 *     then out = old + y in accumulate mode.  No FMA contraction, no
 *     flush-to-zero.  Results are bitwise independent of CTA budget, chunk
 *     size, stage shape and scheduling.
 */
#ifndef TIDE_H
#define TIDE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TIDE_API __attribute__((visibility("default")))
#else
#define TIDE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TIDE_OK = 0,
    TIDE_ERR_INVALID_ARG = 1,  /* bad count, size, null pointer, aliasing, ... */
    TIDE_ERR_ALIGNMENT = 2,    /* pointer not aligned to its element size */
    TIDE_ERR_UNSUPPORTED = 3,  /* valid request this build does not implement: fall back to the two-pass path */
    TIDE_ERR_OOM = 4,          /* plan tables could not be allocated */
    TIDE_ERR_CUDA = 5,         /* a CUDA runtime call failed (detail in tide_last_error) */
    TIDE_ERR_TIMEOUT = 6       /* a bounded device-side wait expired (tide_last_device_status) */
} tide_status_t;

/* Opaque plan: geometry, work list and device tables of one parameter group. */
typedef struct tide_plan tide_plan_t;

/* One parameter of the group (Section 2.1 notation). */
typedef struct {
    /* Host array of W pointers: rank_base[u] is G_p^(u), the gradient of
     * this parameter on virtual rank u (bf16, or fp32 with TIDE_DTYPE_F32),
     * row-major and contiguous (dim0 * row_numel elements).  Each points to
     * memory of the current device, managed memory, or page-locked host
     * memory mapped into the device's address space at the same address
     * (cudaHostAlloc; cudaHostRegister where the device uses host pointers):
     * gradients in host memory are read in place over the host link
     * (NVLink-C2C on Grace systems) by the direct-load kernel.  Pageable host
     * memory is refused.  Aligned to the element size; 16-byte alignment
     * enables the vector and bulk-copy paths.  The array itself is copied
     * during the call. */
    const void *const *rank_base;
    int64_t dim0;          /* D_p >= 0: extent of dimension 0 (0 = empty tensor, pointers may be NULL) */
    int64_t row_numel;     /* K_p >= 0: product of the trailing dimensions (1 for a vector) */
    int64_t shard_offset;  /* o_p in elements inside a rank slot, or -1 to use the prefix sum
                              of the preceding parameters' R_q K_q.  Explicit offsets must not
                              make two shards overlap. */
} tide_param_desc_t;

/* Summation order of the reduce-scatter fold (Section 4.3).  Every order is
 * deterministic (bitwise reproducible for a plan); orders other than rank
 * order differ from it by rounding only (within 1e-6 of it in the max-norm
 * on the benchmark workloads). */
enum {
    TIDE_ORDER_RANK_ASC = 0,   /* ((G0 + G1) + G2) + ... : the bit-exact contract */
    TIDE_ORDER_STAGED_OWN = 1, /* one node (Level 1): every rank except the destination r in
                                  ascending order, then r's own contribution */
    TIDE_ORDER_NODES = 2,      /* two levels: W = M nodes of node_size ranks; each node's partial
                                  adds its ranks except n*node_size + (r mod node_size) in
                                  ascending order, then that rank; the node partials are then
                                  added in node order */
    TIDE_ORDER_TREE = 3        /* pairwise summation of ranks 0..W-1: neighbours added level by
                                  level, an odd last value carried up (depth ceil(log2 W)).  Not
                                  one of the paper's orders: the balanced alternative to its
                                  chains.  Bulk kernel; stage fills of a power-of-two number of
                                  ranks, at most 255 full fills per chunk (W / fill_ranks) */
};

/* Work distribution of the fold's persistent grid (bitwise identical results). */
enum {
    TIDE_SCHED_AUTO = 0,     /* the library's default: TIDE_SCHED_DYNAMIC, or TIDE_SCHED_STATIC
                                when every CTA of the grid gets at most one work item */
    TIDE_SCHED_DYNAMIC = 1,  /* CTAs claim items from a device counter that resets itself (bulk
                                kernel: the producer lane claims each item and posts it to the
                                CTA's consumer warps), so faster SMs take more items: 2-6% faster
                                than TIDE_SCHED_STATIC on the benchmark groups.  The counter
                                lives in the plan, so one plan's folds must not overlap */
    TIDE_SCHED_PER_ITEM = 2, /* one short-lived CTA per work item (the grid is the work list; needs
                                cta_budget 0), as the placement kernel always launches.  Alone it
                                runs about as fast as the persistent grid; with the plan's stream at
                                a lower priority than concurrent compute, the block scheduler hands
                                SMs to the compute kernels as these CTAs retire, so the fold yields
                                without a fixed CTA budget (Section 2.2's SM interference) */
    TIDE_SCHED_STATIC = 3    /* work item i goes to CTA i mod grid */
};

/* Reduce-scatter kernel family. */
enum {
    TIDE_KERNEL_AUTO = 0,    /* the library's default: BULK */
    TIDE_KERNEL_DIRECT = 1,  /* 16-byte vector loads of the W rank rows straight into registers */
    TIDE_KERNEL_BULK = 2     /* warp-specialised: bulk async copies (cp.async.bulk + mbarrier)
                                stage the W rank rows in shared memory */
};

/* All-gather placement engines. */
enum {
    TIDE_AG_SM = 0,      /* placement kernel: 16-byte vector copies per (parameter, rank) piece,
                            one short CTA per 16,384-element work item */
    TIDE_AG_CE_2D = 1,   /* copy engines: one 2D copy per parameter over its full-shard ranks
                            (source pitch = slot stride, destination pitch = R_p K_p) + 1 tail copy;
                            pieces of 1 MiB or more are copied one by one instead, and large 2D
                            copies are split by rows to balance the copy-engine streams */
    TIDE_AG_CE_1D = 2    /* copy engines: one 1D copy per (parameter, rank) piece */
};

/* Gradient element type (b_grad of Section 2.1). */
enum {
    TIDE_DTYPE_BF16 = 0,  /* widened exactly to fp32 */
    TIDE_DTYPE_F32 = 1    /* fp32 gradients, summed as they are */
};

/* Debug bits. */
#define TIDE_DEBUG_HOST_ONLY 0x1u  /* build geometry and work list only: no device tables, no CUDA calls.
                                      Such a plan can be inspected but not launched. */
#define TIDE_DEBUG_SHORT_WAIT 0x2u /* bulk kernel: bound each device-side wait by 50 ms instead of 4 s */
#define TIDE_DEBUG_SKIP_FILL 0x4u  /* bulk kernel: the CTA that takes work item 0 never fills that
                                      item's first stage, so its consumers' bounded wait expires;
                                      exercises the TIMEOUT status path (whatever the schedule).  The
                                      output of that fold is incomplete. */

typedef struct {
    int32_t cta_budget;   /* CTAs of the fold's persistent grid; 0 = one wave at full occupancy (two
                             bulk CTAs per SM).  A budget of at most the SM count gives each bulk
                             CTA an SM: a 192 KB ring and, except in the tree order, 8 consumer
                             warps and 16 KB copies per rank (the fastest shape per SM).  Next to
                             a clustered GEMM, tide_corun_cta_budget gives the budget that keeps
                             the GEMM in one wave */
    int32_t chunk_bytes;  /* bf16 bytes per rank in one work item (multiple of 256); 0 = default */
    int32_t order;        /* TIDE_ORDER_* */
    int32_t sched;        /* TIDE_SCHED_* */
    int32_t kernel;       /* TIDE_KERNEL_* */
    int32_t grad_dtype;   /* TIDE_DTYPE_* */
    uint32_t debug;       /* TIDE_DEBUG_* bits */
    int32_t fill_bytes;   /* bulk kernel: gradient bytes per rank in one shared-memory stage fill
                             (multiple of 16, at most 16384); 0 = 4096, or 16384 when each CTA
                             has an SM (see cta_budget).  A fill holds at most 2,048 elements
                             (8,192 with an SM per CTA; 1,024 for the tree order with 8 or more
                             full fills per chunk), and two stages must fit in shared memory */
    int32_t fill_ranks;   /* bulk kernel: ranks per stage fill (0 = min(W, 8), or min(W, 4) with
                             an SM per CTA); wider groups take
                             several fills per chunk, summed in registers in the plan's order.
                             TIDE_ORDER_TREE: at most 8, rounded down to a power of two when
                             below W, and W / fill_ranks <= 255 */
    int32_t node_size;    /* TIDE_ORDER_NODES: ranks per node, dividing the world; else 0 */
    int32_t ce_streams;   /* copy-engine placement: internal streams the copies are spread over,
                             so several copy engines work at once (0 = 8, at most 8) */
    int32_t reserved[1];  /* must be zero */
} tide_plan_flags_t;

/* Read-only view of one (parameter, rank) shard piece of a plan. */
typedef struct {
    int32_t param;       /* p */
    int32_t rank;        /* r */
    int64_t src_elem;    /* first element of rank r's rows in G_p^(u): r * R_p * K_p */
    int64_t dst_elem;    /* o_p: element offset of the piece inside rank r's slot */
    int64_t n_valid;     /* v_{p,r} * K_p real elements */
    int64_t n_pad;       /* (R_p - v_{p,r}) * K_p padding elements */
} tide_segment_t;

/*
 * Build a plan for one parameter group of `num_params` parameters sharded over
 * `world` virtual ranks (1 <= world <= 1024).  Computes R_p, o_p, S and the
 * P*W shard pieces (Section 2.1), splits them into work items, validates
 * every descriptor, queries the memory kind of every gradient pointer
 * (cudaPointerGetAttributes, about 1 us each), allocates the plan's device
 * tables and uploads them with asynchronous copies on `stream`.  `params` is
 * a host array; `flags` may be NULL for defaults.  On success *plan_out owns
 * the tables.
 * Errors: INVALID_ARG (world, counts, dims, null pointers, overlapping
 * explicit offsets, nonzero reserved fields, node_size not dividing world,
 * a gradient in pageable host memory or in another device's memory),
 * ALIGNMENT (a gradient pointer not aligned to its element size),
 * UNSUPPORTED (a combination this build lacks: orders other than rank order
 * and fp32 gradients run on the bulk kernel only; gradients in host memory
 * take the direct-load kernel, so bf16 in rank order only),
 * OOM, CUDA.
 */
TIDE_API tide_status_t tide_plan_build(int32_t world, int32_t num_params, const tide_param_desc_t *params,
                              const tide_plan_flags_t *flags, void *stream, tide_plan_t **plan_out);

/*
 * Point an existing plan at new gradient storage with the same geometry (for
 * example, the next step's gradients).  dim0, row_numel and shard_offset must
 * equal the plan's, and the gradients must stay in the same kind of memory
 * (device or host) as at build; only pointers that changed are queried
 * again.  The new pointer table is uploaded on `stream`, ordered after
 * earlier work on that stream.
 */
TIDE_API tide_status_t tide_plan_rebind(tide_plan_t *plan, const tide_param_desc_t *params, void *stream);

/*
 * Reduce-scatter fold (Section 4, Equation (5)) of every parameter into every
 * virtual rank's fp32 shard.
 *   out_base: device fp32, W rank slots; rank r's slot starts at
 *             out_base + r * out_slot_stride and its shard of parameter p at
 *             offset o_p.  Padding positions receive alpha * (+0) (or old +
 *             alpha * (+0) in accumulate mode).  Elements of a slot past S are
 *             not touched.  4-byte aligned.  Must not overlap any gradient.
 *   out_slot_stride: elements between rank slots, >= S.
 *   alpha: scale applied to the fp32 sum (1/W for an average).
 *   accumulate: 0 = overwrite, 1 = add into the existing shard values.
 * Enqueued on `stream`; returns without waiting.
 */
TIDE_API tide_status_t tide_rs_fold(tide_plan_t *plan, float *out_base, int64_t out_slot_stride, float alpha,
                           int32_t accumulate, void *stream);

/*
 * All-gather placement (Section 2.1, Equation (2)).
 *   slots_base: device bf16, W rank slots of `slot_stride` elements (>= S);
 *               rank r's shard of parameter p is read from
 *               slots_base + r * slot_stride + o_p.  Padding is never read.
 *   full: host array of P device pointers; full[p] receives parameter p as a
 *         contiguous row-major (dim0, row_numel) bf16 tensor.  2-byte aligned;
 *         must not overlap the slots or each other.
 *   mode: TIDE_AG_SM, TIDE_AG_CE_2D or TIDE_AG_CE_1D.
 * Bitwise copy; enqueued on `stream`.
 */
TIDE_API tide_status_t tide_ag_place(tide_plan_t *plan, const void *slots_base, int64_t slot_stride, void *const *full,
                            int32_t mode, void *stream);

/*
 * Mixed-precision all-gather placement (Section 3.1: groups that keep fp32
 * master shards cast them to bf16 for the all-gather; here the cast is fused
 * into the placement of Eq. (2)).
 *   slots_base: device fp32, W rank slots of `slot_stride` elements (>= S);
 *               4-byte aligned.  Padding is never read.
 *   full: as tide_ag_place; each element is the fp32 value rounded to the
 *         nearest bf16 (ties to even; NaN stays NaN, overflow gives +-inf).
 * SM kernel only (copy engines cannot convert).  Enqueued on `stream`.
 */
TIDE_API tide_status_t tide_ag_place_f32(tide_plan_t *plan, const float *slots_base, int64_t slot_stride,
                                         void *const *full, void *stream);

/* Free the plan's device tables after synchronising the stream of its last use. */
TIDE_API tide_status_t tide_plan_destroy(tide_plan_t *plan);

/* S: elements per rank slot (the smallest valid out_slot_stride / slot_stride); -1 for NULL. */
TIDE_API int64_t tide_plan_slot_numel(const tide_plan_t *plan);

/* Number of (parameter, rank) shard pieces, P * W; -1 for NULL. */
TIDE_API int64_t tide_plan_num_segments(const tide_plan_t *plan);

/* Copy shard piece `index` (ordered by parameter, then rank) into *out. */
TIDE_API tide_status_t tide_plan_segment(const tide_plan_t *plan, int64_t index, tide_segment_t *out);

/* Launch geometry the plan will use for the fold: grid CTAs, threads per CTA,
 * work items, elements per item.  Any pointer may be NULL. */
TIDE_API tide_status_t tide_plan_fold_config(const tide_plan_t *plan, int32_t *grid, int32_t *block, int64_t *items,
                                    int64_t *chunk_elems);

/*
 * Read and clear the plan's device status word (synchronises `stream`).
 * Returns TIDE_ERR_TIMEOUT if a bounded device-side wait of an earlier fold
 * on this plan expired (that fold's output is then incomplete), else TIDE_OK.
 * With plan = NULL, reads and clears the status word of the allocation-free
 * fold (tide_rs_fold_noalloc) on the current device instead: TIDE_ERR_TIMEOUT
 * if a wait of any of its folds there expired since the last such read
 * (TIDE_OK if that entry point never ran on the device).  Neither form
 * allocates device memory.
 */
TIDE_API tide_status_t tide_last_device_status(tide_plan_t *plan, void *stream);

/* Kernels this library has launched in this process (all plans, all calls). */
TIDE_API uint64_t tide_launch_count(void);

/*
 * Allocation-free reduce-scatter fold, for callers that cannot allocate GPU
 * memory.  The paper has no counterpart to this entry point.
 *
 * tide_plan_build allocates device tables with cudaMalloc.  Callers that run
 * inside an allocator (an allocation hook or an out-of-memory handler), under
 * a memory pool or cap that forbids new device allocations, or that must not
 * leave allocations behind can use this call instead: it computes the same
 * result as tide_plan_build + tide_rs_fold + tide_plan_destroy with default
 * flags (bit for bit, and equal to Equation (5) in rank order), but keeps its
 * tables in one fixed device array owned by the library and calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   Arguments: as tide_plan_build's (world, num_params, params) followed by
 *   tide_rs_fold's (out_base, out_slot_stride, alpha, accumulate, stream);
 *   S is computed from params the same way; explicit shard offsets must be
 *   given in increasing order (each at least the previous shard's end).  The
 *   gradients must be device (or managed) memory of the current device: this
 *   entry point does not query pointer kinds and always runs the bulk-copy
 *   kernel, so gradients in host memory take tide_plan_build.
 *   Limit: the call's tables (8 bytes per gradient pointer, 48 per
 *   (parameter, rank) piece, 16 per work item of 8,192 elements, plus
 *   alignment) must fit in TIDE_NOALLOC_SCRATCH_BYTES; larger requests return
 *   TIDE_ERR_INVALID_ARG without doing anything.  All five of this library's
 *   benchmark workloads fit (the largest needs about 2 MB).
 *   Memory: the array occupies TIDE_NOALLOC_SCRATCH_BYTES on each GPU where
 *   the library is used, until the process exits.
 *   Set-up: the first call on each device looks up the array's device address
 *   with that device current and loads the fold kernels (the runtime may
 *   reserve device memory for them then); make that first call before any
 *   stream capture and outside the context that cannot allocate.  A call with
 *   num_params = 0 does only this set-up.  Later calls on the device allocate
 *   nothing.
 *   Errors: as tide_plan_build and tide_rs_fold; nothing is enqueued on
 *   failure.  A bounded device-side wait that expires is recorded in the
 *   array's status word, which later calls leave as it is:
 *   tide_last_device_status(NULL, stream) reads and clears it.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   tables and the schedule's work counter.  Calls that overlap on the GPU
 *   (different streams without an ordering between them) race; calls on one
 *   stream are ordered.  Calls from several host threads are serialised by a
 *   lock.
 */
#define TIDE_NOALLOC_SCRATCH_BYTES ((size_t)4 * 1024 * 1024)
TIDE_API tide_status_t tide_rs_fold_noalloc(int32_t world, int32_t num_params, const tide_param_desc_t *params,
                                            float *out_base, int64_t out_slot_stride, float alpha,
                                            int32_t accumulate, void *stream);

/* ------------------------------------------------------------------------
 * Multi-node schedule planners (host only).  A single GPU runs none of these
 * schedules; a multi-node runtime plans with them.
 * ---------------------------------------------------------------------- */

/* Section 4.2, Equations (6)-(8): for destination node m and contributor
 * node n of M nodes with L GPUs each, the send-order contributor index is
 * c = (m - n) mod M (n != m) or M (own node), and its partial for sub-slice s
 * lands in inbox block s of destination GPU (s - c mod M) mod L.  Returns that
 * GPU, or -1 for arguments out of range. */
TIDE_API int32_t tide_latin_square_gpu(int32_t s, int32_t m, int32_t n, int32_t M, int32_t L);

typedef struct {
    int32_t waves;          /* ceil(M / w_wave) */
    int32_t generations;    /* inbox buffer generations: 1 for one wave or me = 1, else 2 */
    int32_t network_rounds; /* sum over waves of ceil(remote contributors of the wave / k) */
    int32_t zero_blocks;    /* stale inbox blocks zeroed before landings, whole schedule */
} tide_wave_plan_t;

/* Appendix D base-plan check for (M, L, w_wave, k, me): contributors 1..M in
 * increasing order, w_wave per wave, k concurrent rail transfers per round,
 * me = 1 for the memory-efficient single-generation inbox.  TIDE_OK when every
 * wave is collision-free (Proposition 4.1 guarantees it when w_wave divides
 * L); TIDE_ERR_UNSUPPORTED when two contributors of a wave would land on the
 * same GPU (the plan must be rejected); INVALID_ARG for M < 1, L outside
 * [1, 64], w_wave < 1, k < 1 or a bad me. */
TIDE_API tide_status_t tide_rs_wave_plan(int32_t M, int32_t L, int32_t w_wave, int32_t k, int32_t me,
                                         tide_wave_plan_t *out);

/* Stale blocks to zero before landing `wave`: blocks the previous wave on the
 * same buffer generation wrote that this wave does not.  zero_mask[j] bit s
 * set = zero block s of GPU j (host array of L entries). */
TIDE_API tide_status_t tide_rs_wave_zero_mask(int32_t M, int32_t L, int32_t w_wave, int32_t me, int32_t wave,
                                              uint64_t *zero_mask);

/* Section 3.1: recursive doubling over M nodes.  Writes, for each round d,
 * count[d] = min(2^d, M - 2^d) shards forwarded to (n - 2^d) mod M and
 * step[d] = 2^d; returns the number of rounds ceil(log2 M), or -1 if M < 1 or
 * max_rounds is too small. */
TIDE_API int32_t tide_bruck_schedule(int32_t M, int32_t *count, int32_t *step, int32_t max_rounds);

/* ------------------------------------------------------------------------
 * Diagnostics
 * ---------------------------------------------------------------------- */

/* SM-id probe (the measurement of Table 5 / Figure 3): launches `ctas` CTAs
 * of 128 threads in clusters of `cluster` (1..8), each with `smem_bytes` of
 * dynamic shared memory (enough to fill an SM keeps one CTA per SM).  Each
 * CTA writes smid[i] (the SM it ran on) and t_in[i] / t_out[i] (%globaltimer
 * nanoseconds at entry and exit) and holds its SM for hold_ns (at most 10 ms;
 * the wait is bounded by time).  Outputs are device arrays of `ctas` entries.
 * If t_ready (device, one entry) is not NULL, a one-thread kernel launched
 * just before the probe on the same stream writes the time the stream
 * reached the probe, so that entry delays (blocked CTAs) can be measured.
 * Enqueued on `stream`. */
TIDE_API tide_status_t tide_sm_probe(int32_t ctas, int32_t cluster, int32_t smem_bytes, uint64_t hold_ns,
                                     uint32_t *smid, uint64_t *t_in, uint64_t *t_out, uint64_t *t_ready,
                                     void *stream);

/* Clusters of the probe's shape the current device can hold at once
 * (its "cluster slots"), or -1. */
TIDE_API int32_t tide_sm_probe_max_clusters(int32_t cluster, int32_t smem_bytes);

/*
 * CTA budget for a fold that runs next to a clustered GEMM (Section 2.2,
 * Equation (4): T_gemm ~ ceil(n_gemm / (n_slot - n_blk)) T_wave).  A GEMM of
 * gemm_ctas CTAs in clusters of `cluster` CTAs has n_gemm = ceil(gemm_ctas /
 * cluster) clusters; the device holds cluster_slots (n_slot, from
 * tide_sm_probe_max_clusters with the GEMM's cluster size and per-CTA shared
 * memory) of them at once.  The GEMM keeps a single wave while the fold blocks
 * at most n_slot - n_gemm slots, so the budget is (n_slot - n_gemm) * cluster:
 * fold CTAs with an SM each (any budget up to the SM count), filling that
 * many spare slots.  Pass the result as tide_plan_flags_t.cta_budget.
 * Host arithmetic only (no CUDA call).  Returns 0 when the GEMM needs every
 * slot (then every resident fold CTA can push GEMM CTAs into a second wave),
 * -1 for arguments out of range (any count < 1, cluster > 16).
 * Example: GB300 holds 36 clusters of four 213 KB CTAs; the 256 x 8192 x 8192
 * GEMM's 128 CTAs form 32, so the budget is (36 - 32) * 4 = 16 CTAs.
 */
TIDE_API int32_t tide_corun_cta_budget(int32_t cluster_slots, int32_t gemm_ctas, int32_t cluster);

/* Human-readable name of a status code. */
TIDE_API const char *tide_status_string(tide_status_t status);

/* Detail message of the last failing call on this thread ("" if none). */
TIDE_API const char *tide_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TIDE_H */

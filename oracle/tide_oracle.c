/*
 * CPU oracle for the FSDP2 layout-folded reduce-scatter and all-gather
 * placement described in "The Endgame of FSDP Communication: Layout-Aware
 * Collectives on Copy Engines, RDMA, and NVSwitch" (TIDE).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or table with the CUDA library.
 *
 * Plain, slow and single-threaded on purpose.  Build with
 *   gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * so that every float operation below is one IEEE binary32 operation with
 * round-to-nearest-even (no FMA contraction, no flush-to-zero).
 *
 * Notation follows Section 2.1 / Table 2 of the paper, with W for the number
 * of (virtual) ranks the paper calls N:
 *   D_p  dim-0 extent of parameter p,   K_p  product of its trailing dims,
 *   R_p  = ceil(D_p / W) padded rows per rank,
 *   o_p  = sum_{q<p} R_q K_q  (prefix offset, in elements),
 *   S    = sum_p R_p K_p      (elements per rank slot).
 * Rank r owns rows [r R_p, (r+1) R_p) of parameter p; rows past D_p are zero
 * (Section 2.1, "The backward reduce-scatter boundary").  The number of real
 * rows rank r holds is therefore v_{p,r} = clamp(D_p - r R_p, 0, R_p).
 *
 * Parity pins: every function here is pinned by the CPU tests (brute force on
 * tiny shapes, torch.chunk / torch._chunk_cat library equivalence, exact
 * integer sums, a closed-form summation-order probe, fp64 error bounds,
 * special values and hand-worked fixtures).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

/* Exact widening of a bf16 bit pattern: bf16 is the top half of binary32. */
static float bf16_to_f32(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/* Section 2.1: padded per-rank rows R_p = ceil(D_p / W) and the prefix
 * offsets o_p of the parameter-major concatenation inside one rank slot. */
int oracle_geometry(int32_t world, int32_t nparams, const int64_t *dim0, const int64_t *row_numel,
                    int64_t *rows_per_rank, int64_t *shard_offset, int64_t *slot_numel)
{
    if (world < 1 || nparams < 0)
        return ORACLE_EINVAL;
    int64_t off = 0;
    for (int32_t p = 0; p < nparams; ++p) {
        if (dim0[p] < 0 || row_numel[p] < 0)
            return ORACLE_EINVAL;
        int64_t R = (dim0[p] + world - 1) / world;
        rows_per_rank[p] = R;
        shard_offset[p] = off;
        off += R * row_numel[p];
    }
    *slot_numel = off;
    return ORACLE_OK;
}

/* Real (unpadded) rows of parameter p that rank r holds. */
int64_t oracle_valid_rows(int64_t dim0, int64_t rows_per_rank, int32_t r)
{
    int64_t v = dim0 - (int64_t)r * rows_per_rank;
    if (v < 0)
        v = 0;
    if (v > rows_per_rank)
        v = rows_per_rank;
    return v;
}

/*
 * Equations (3) and (5) for one window of one destination shard.
 *
 * src[u] points at the first real element of the window in source rank u's
 * gradient; the window holds n_valid real elements followed by n_pad padding
 * elements (rows past D_p).
 *
 * Pass 1 (Eq. 3, FSDP2's pack): each source rank's contribution is sliced,
 * zero-padded and widened to fp32 into its own buffer.
 * Pass 2 (Eq. 5): the W buffers are added in rank order 0, 1, ..., W-1,
 * starting from rank 0's value, in fp32; the sum is scaled by alpha and, in
 * accumulate mode, added to the existing shard value.
 *
 * old may equal out (in-place accumulate).  Returns ORACLE_ENOMEM if the
 * pack buffer cannot be allocated.
 */
int oracle_rs_window(int32_t world, int64_t n_valid, int64_t n_pad, const uint16_t *const *src,
                     float alpha, int32_t accumulate, const float *old, float *out)
{
    int64_t n = n_valid + n_pad;
    if (world < 1 || n_valid < 0 || n_pad < 0)
        return ORACLE_EINVAL;
    if (n == 0)
        return ORACLE_OK;
    float *pack = (float *)malloc((size_t)world * (size_t)n * sizeof(float));
    if (!pack)
        return ORACLE_ENOMEM;

    /* pass 1: slice, zero-pad, upcast */
    for (int32_t u = 0; u < world; ++u) {
        float *dst = pack + (size_t)u * (size_t)n;
        for (int64_t j = 0; j < n_valid; ++j)
            dst[j] = bf16_to_f32(src[u][j]);
        for (int64_t j = n_valid; j < n; ++j)
            dst[j] = 0.0f;
    }

    /* pass 2: rank-ordered fp32 reduction, scale, optional accumulate */
    for (int64_t j = 0; j < n; ++j) {
        float acc = pack[j];
        for (int32_t u = 1; u < world; ++u)
            acc = acc + pack[(size_t)u * (size_t)n + (size_t)j];
        float y = alpha * acc;
        out[j] = accumulate ? old[j] + y : y;
    }
    free(pack);
    return ORACLE_OK;
}

/*
 * Full reduce-scatter of one parameter group (Eq. 5 for every p and r).
 *
 * grads[p * world + u] points at parameter p's full gradient on source rank
 * u, row-major (D_p, K_p) bf16 bits.  out is W rank slots of `stride`
 * elements each (stride >= S); rank r's shard of p lands at
 * out[r * stride + o_p].  Elements of a slot past S are not touched.
 */
int oracle_rs(int32_t world, int32_t nparams, const int64_t *dim0, const int64_t *row_numel,
              const uint16_t *const *grads, float alpha, int32_t accumulate, float *out, int64_t stride)
{
    int64_t *R = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    int64_t *o = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    const uint16_t **src = (const uint16_t **)malloc(sizeof(uint16_t *) * (size_t)world);
    int64_t S = 0;
    int rc = ORACLE_OK;
    if (!R || !o || !src) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    rc = oracle_geometry(world, nparams, dim0, row_numel, R, o, &S);
    if (rc != ORACLE_OK)
        goto done;
    if (stride < S) {
        rc = ORACLE_EINVAL;
        goto done;
    }
    for (int32_t p = 0; p < nparams && rc == ORACLE_OK; ++p) {
        int64_t K = row_numel[p];
        for (int32_t r = 0; r < world && rc == ORACLE_OK; ++r) {
            int64_t v = oracle_valid_rows(dim0[p], R[p], r);
            for (int32_t u = 0; u < world; ++u)
                src[u] = grads[(size_t)p * (size_t)world + (size_t)u] + (size_t)r * (size_t)R[p] * (size_t)K;
            float *dst = out + (size_t)r * (size_t)stride + (size_t)o[p];
            rc = oracle_rs_window(world, v * K, (R[p] - v) * K, src, alpha, accumulate, dst, dst);
        }
    }
done:
    free(R);
    free(o);
    free((void *)src);
    return rc;
}

/*
 * All-gather placement (Section 2.1, Eq. 2): rank r's shard of p sits in the
 * rank-major input at slot r, offset o_p; its i-th real row becomes row
 * r R_p + i of the full (D_p, K_p) tensor.  Padding rows are dropped.
 *
 * slots is W rank slots of `stride` bf16 elements; full[p] is parameter p's
 * output tensor.
 */
int oracle_ag(int32_t world, int32_t nparams, const int64_t *dim0, const int64_t *row_numel,
              const uint16_t *slots, int64_t stride, uint16_t *const *full)
{
    int64_t *R = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    int64_t *o = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    int64_t S = 0;
    int rc = ORACLE_OK;
    if (!R || !o) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    rc = oracle_geometry(world, nparams, dim0, row_numel, R, o, &S);
    if (rc != ORACLE_OK)
        goto done;
    if (stride < S) {
        rc = ORACLE_EINVAL;
        goto done;
    }
    for (int32_t p = 0; p < nparams; ++p) {
        int64_t K = row_numel[p];
        for (int32_t r = 0; r < world; ++r) {
            int64_t v = oracle_valid_rows(dim0[p], R[p], r);
            for (int64_t i = 0; i < v; ++i) {
                const uint16_t *from = slots + (size_t)r * (size_t)stride + (size_t)o[p] + (size_t)(i * K);
                uint16_t *to = full[p] + (size_t)((r * R[p] + i) * K);
                for (int64_t k = 0; k < K; ++k)
                    to[k] = from[k];
            }
        }
    }
done:
    free(R);
    free(o);
    return rc;
}

/*
 * Round-to-nearest-even narrowing of a binary32 value to bf16 (8 significant
 * bits), written from the definition: keep the upper 16 bits, then look at
 * the 16 discarded bits -- above one half of the last kept place round up,
 * below it truncate, exactly one half round to the even neighbour.  A carry
 * out of the mantissa moves into the exponent, which turns the largest finite
 * values into infinity as IEEE rounding requires.  NaN stays NaN (quiet, same
 * sign).
 */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t w;
    memcpy(&w, &x, sizeof w);
    if ((w & 0x7F800000u) == 0x7F800000u && (w & 0x007FFFFFu) != 0)
        return (uint16_t)((w >> 16) | 0x0040u);
    uint32_t kept = w >> 16;
    uint32_t dropped = w & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/*
 * Mixed-precision all-gather placement (Section 3.1: mixed-precision groups
 * keep fp32 master shards and cast them to bf16 for the all-gather): the
 * placement of Eq. (2) reading fp32 rank slots and writing each element
 * rounded to bf16.  slots is W rank slots of `stride` fp32 elements.
 */
int oracle_ag_cast(int32_t world, int32_t nparams, const int64_t *dim0, const int64_t *row_numel,
                   const float *slots, int64_t stride, uint16_t *const *full)
{
    int64_t *R = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    int64_t *o = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    int64_t S = 0;
    int rc = ORACLE_OK;
    if (!R || !o) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    rc = oracle_geometry(world, nparams, dim0, row_numel, R, o, &S);
    if (rc != ORACLE_OK)
        goto done;
    if (stride < S) {
        rc = ORACLE_EINVAL;
        goto done;
    }
    for (int32_t p = 0; p < nparams; ++p) {
        int64_t K = row_numel[p];
        for (int32_t r = 0; r < world; ++r) {
            int64_t v = oracle_valid_rows(dim0[p], R[p], r);
            for (int64_t i = 0; i < v; ++i) {
                const float *src_row = slots + (size_t)r * (size_t)stride + (size_t)o[p] + (size_t)(i * K);
                uint16_t *dst_row = full[p] + (size_t)((r * R[p] + i) * K);
                for (int64_t k = 0; k < K; ++k)
                    dst_row[k] = oracle_f32_to_bf16(src_row[k]);
            }
        }
    }
done:
    free(R);
    free(o);
    return rc;
}

/* ------------------------------------------------------------------------
 * Summation orders other than rank order, and fp32 gradients.
 *
 * Section 4.3: Level 1 adds the L - 1 staged contributions in local-rank
 * order and then the owner's own contribution, in fp32; Level 2 adds the
 * node partials.  Orders (readings of that section for virtual ranks):
 *   ORACLE_ORDER_RANK      ((G0 + G1) + G2) + ...            (rank order)
 *   ORACLE_ORDER_STAGED    one node: every rank except the destination r in
 *                          ascending order, then r's own contribution
 *   ORACLE_ORDER_NODES     W = M L ranks in M nodes of L: node n's partial is
 *                          its ranks except n L + (r mod L) ascending, then
 *                          that rank; the M node partials are then added in
 *                          node order
 *   ORACLE_ORDER_TREE      pairwise (balanced-tree) summation of the rank
 *                          sequence 0..W-1: level by level, neighbours
 *                          (2i, 2i+1) are added and an odd last value moves
 *                          up unchanged, until one value is left.  The page
 *                          names no tree order; this is the textbook pairwise
 *                          summation, whose rounding error grows with
 *                          ceil(log2 W) instead of W - 1.
 * dtype 0: bf16 gradients (widened exactly); dtype 1: fp32 gradients
 * (b_grad = 4, used as they are).
 * ---------------------------------------------------------------------- */
#define ORACLE_ORDER_RANK 0
#define ORACLE_ORDER_STAGED 1
#define ORACLE_ORDER_NODES 2
#define ORACLE_ORDER_TREE 3

static float widen(const void *src, int32_t dtype, int64_t j)
{
    if (dtype == 0)
        return bf16_to_f32(((const uint16_t *)src)[j]);
    return ((const float *)src)[j];
}

/* The order in which the W contributions to destination rank r are added
 * (seq), and how many consecutive entries form one partial (group; the
 * partials are then added in sequence order). */
static int make_sequence(int32_t world, int32_t order, int32_t node_size, int32_t r, int32_t *seq, int32_t *group)
{
    if (order == ORACLE_ORDER_RANK || order == ORACLE_ORDER_TREE) {
        for (int32_t u = 0; u < world; ++u)
            seq[u] = u;
        *group = world;
        return ORACLE_OK;
    }
    if (order == ORACLE_ORDER_STAGED) {
        int32_t q = 0;
        for (int32_t u = 0; u < world; ++u)
            if (u != r)
                seq[q++] = u;
        seq[q] = r;
        *group = world;
        return ORACLE_OK;
    }
    if (order == ORACLE_ORDER_NODES) {
        if (node_size < 1 || world % node_size != 0)
            return ORACLE_EINVAL;
        int32_t q = 0;
        for (int32_t n = 0; n < world / node_size; ++n) {
            int32_t owner = n * node_size + r % node_size;
            for (int32_t l = 0; l < node_size; ++l)
                if (n * node_size + l != owner)
                    seq[q++] = n * node_size + l;
            seq[q++] = owner;
        }
        *group = node_size;
        return ORACLE_OK;
    }
    return ORACLE_EINVAL;
}

/* Eq. (3) + Eq. (5) for one window of destination rank `dest`, in `order`. */
int oracle_rs_window_ex(int32_t world, int32_t dtype, int32_t order, int32_t node_size, int32_t dest,
                        int64_t n_valid, int64_t n_pad, const void *const *src, float alpha, int32_t accumulate,
                        const float *old, float *out)
{
    int64_t n = n_valid + n_pad;
    if (world < 1 || n_valid < 0 || n_pad < 0 || (dtype != 0 && dtype != 1) || dest < 0 || dest >= world)
        return ORACLE_EINVAL;
    if (n == 0)
        return ORACLE_OK;
    int32_t *seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)world);
    float *pack = (float *)malloc((size_t)world * (size_t)n * sizeof(float));
    float *level = (float *)malloc(sizeof(float) * (size_t)world);
    int32_t group = world;
    int rc = (seq && pack && level) ? make_sequence(world, order, node_size, dest, seq, &group) : ORACLE_ENOMEM;
    if (rc != ORACLE_OK)
        goto done;
    /* pass 1: slice, zero-pad, widen */
    for (int32_t u = 0; u < world; ++u) {
        float *dst = pack + (size_t)u * (size_t)n;
        for (int64_t j = 0; j < n_valid; ++j)
            dst[j] = widen(src[u], dtype, j);
        for (int64_t j = n_valid; j < n; ++j)
            dst[j] = +0.0f;
    }
    /* pass 2: partials of `group` consecutive contributions of the sequence,
     * then the partials in sequence order; or the pairwise tree */
    for (int64_t j = 0; j < n; ++j) {
        float total = 0.0f;
        if (order == ORACLE_ORDER_TREE) {
            int32_t m = world;
            for (int32_t q = 0; q < world; ++q)
                level[q] = pack[(size_t)seq[q] * (size_t)n + (size_t)j];
            while (m > 1) {
                for (int32_t i = 0; i < m / 2; ++i)
                    level[i] = level[2 * i] + level[2 * i + 1];
                if (m % 2 == 1)
                    level[m / 2] = level[m - 1];
                m = (m + 1) / 2;
            }
            total = level[0];
        } else {
            for (int32_t g0 = 0; g0 < world; g0 += group) {
                float part = pack[(size_t)seq[g0] * (size_t)n + (size_t)j];
                for (int32_t q = g0 + 1; q < g0 + group; ++q)
                    part = part + pack[(size_t)seq[q] * (size_t)n + (size_t)j];
                total = (g0 == 0) ? part : total + part;
            }
        }
        float y = alpha * total;
        out[j] = accumulate ? (old[j] + y) : y;
    }
done:
    free(seq);
    free(pack);
    free(level);
    return rc;
}

/* Full reduce-scatter in `order` with `dtype` gradients (grads[p * world + u]). */
int oracle_rs_ex(int32_t world, int32_t dtype, int32_t order, int32_t node_size, int32_t nparams,
                 const int64_t *dim0, const int64_t *row_numel, const void *const *grads, float alpha,
                 int32_t accumulate, float *out, int64_t stride)
{
    const size_t esz = dtype == 0 ? 2u : 4u;
    int64_t *R = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    int64_t *o = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nparams > 0 ? nparams : 1));
    const void **src = (const void **)malloc(sizeof(void *) * (size_t)world);
    int64_t S = 0;
    int rc = ORACLE_OK;
    if (!R || !o || !src) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    rc = oracle_geometry(world, nparams, dim0, row_numel, R, o, &S);
    if (rc != ORACLE_OK)
        goto done;
    if (stride < S) {
        rc = ORACLE_EINVAL;
        goto done;
    }
    for (int32_t p = 0; p < nparams && rc == ORACLE_OK; ++p) {
        int64_t K = row_numel[p];
        for (int32_t r = 0; r < world && rc == ORACLE_OK; ++r) {
            int64_t v = oracle_valid_rows(dim0[p], R[p], r);
            for (int32_t u = 0; u < world; ++u)
                src[u] = (const char *)grads[(size_t)p * (size_t)world + (size_t)u] +
                         (size_t)r * (size_t)R[p] * (size_t)K * esz;
            float *dst = out + (size_t)r * (size_t)stride + (size_t)o[p];
            rc = oracle_rs_window_ex(world, (int32_t)(esz == 4), order, node_size, r, v * K, (R[p] - v) * K, src,
                                     alpha, accumulate, dst, dst);
        }
    }
done:
    free(R);
    free(o);
    free((void *)src);
    return rc;
}

// Multi-node schedule planners of TIDE (host code only): the Latin-square
// sub-slice placement and wave acceptance of the reduce-scatter's Level 2
// (Section 4.2, Equations (6)-(8), Proposition 4.1, Appendix D) and the
// recursive-doubling rounds of the all-gather (Section 3.1).  A single GPU
// runs none of these schedules; they are exposed so that a multi-node
// runtime can plan with them and are checked exhaustively on the CPU.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "tide_internal.h"

namespace {

constexpr int32_t kMaxNodeGpus = 64;  // L: one 64-bit block mask per GPU

int32_t cbar(int32_t c, int32_t M) { return c % M; }

// Equation (8): destination GPU of contributor c's sub-slice s.
int32_t landing(int32_t s, int32_t c, int32_t M, int32_t L) { return ((s - cbar(c, M)) % L + L) % L; }

bool args_ok(int32_t M, int32_t L, int32_t w_wave) { return M >= 1 && L >= 1 && L <= kMaxNodeGpus && w_wave >= 1; }

}  // namespace

extern "C" {

int32_t tide_latin_square_gpu(int32_t s, int32_t m, int32_t n, int32_t M, int32_t L)
{
    if (M < 1 || L < 1 || s < 0 || s >= L || m < 0 || m >= M || n < 0 || n >= M)
        return -1;
    const int32_t c = n != m ? ((m - n) % M + M) % M : M;  // Equation (6)
    return landing(s, c, M, L);
}

static tide_status_t rs_wave_zero_mask_impl(int32_t M, int32_t L, int32_t w_wave, int32_t me, int32_t wave,
                                            uint64_t *zero_mask);

static tide_status_t rs_wave_plan_impl(int32_t M, int32_t L, int32_t w_wave, int32_t k, int32_t me,
                                       tide_wave_plan_t *out)
{
    tide::record_error("");
    if (!args_ok(M, L, w_wave) || k < 1 || (me != 0 && me != 1) || !out) {
        tide::record_error("need M >= 1, 1 <= L <= 64, w_wave >= 1, k >= 1, me in {0, 1}, out != NULL");
        return TIDE_ERR_INVALID_ARG;
    }
    std::memset(out, 0, sizeof *out);
    const int32_t W = (M + w_wave - 1) / w_wave;
    out->waves = W;
    out->generations = (W == 1 || me) ? 1 : 2;
    // Contributors 1..M in increasing order, w_wave per wave; a wave collides
    // when two of its contributors share c_bar mod L (then they land on the
    // same GPU for every sub-slice s).
    std::vector<int32_t> owner(static_cast<size_t>(L), 0);
    for (int32_t w = 0; w < W; ++w) {
        const int32_t c0 = w * w_wave + 1, c1 = (w + 1) * w_wave < M ? (w + 1) * w_wave : M;
        std::fill(owner.begin(), owner.end(), 0);
        int32_t remote = 0;
        for (int32_t c = c0; c <= c1; ++c) {
            const int32_t j = landing(0, c, M, L);
            if (owner[size_t(j)]) {
                char buf[160];
                snprintf(buf, sizeof buf, "wave %d: contributors %d and %d land on the same GPU (M=%d, L=%d, w_wave=%d)",
                         w, owner[size_t(j)], c, M, L, w_wave);
                tide::record_error(buf);
                return TIDE_ERR_UNSUPPORTED;
            }
            owner[size_t(j)] = c;
            remote += c != M;
        }
        out->network_rounds += (remote + k - 1) / k;
    }
    // Stale inbox blocks over the schedule (zeroed before each landing).
    for (int32_t w = 0; w < W; ++w) {
        std::vector<uint64_t> mask(static_cast<size_t>(L));
        rs_wave_zero_mask_impl(M, L, w_wave, me, w, mask.data());
        for (uint64_t m : mask)
            out->zero_blocks += __builtin_popcountll(m);
    }
    return TIDE_OK;
}

static tide_status_t rs_wave_zero_mask_impl(int32_t M, int32_t L, int32_t w_wave, int32_t me, int32_t wave,
                                            uint64_t *zero_mask)
{
    if (!args_ok(M, L, w_wave) || (me != 0 && me != 1) || !zero_mask) {
        tide::record_error("need M >= 1, 1 <= L <= 64, w_wave >= 1, me in {0, 1}, zero_mask != NULL");
        return TIDE_ERR_INVALID_ARG;
    }
    const int32_t W = (M + w_wave - 1) / w_wave;
    if (wave < 0 || wave >= W) {
        tide::record_error("wave index out of range");
        return TIDE_ERR_INVALID_ARG;
    }
    const int32_t gens = (W == 1 || me) ? 1 : 2;
    // Blocks (gpu j, sub-slice s) written by a wave: each contributor c
    // writes block s on GPU landing(s, c) for every s.
    auto written = [&](int32_t w, std::vector<uint64_t> &m) {
        std::fill(m.begin(), m.end(), 0);
        if (w < 0)
            return;
        const int32_t c0 = w * w_wave + 1, c1 = (w + 1) * w_wave < M ? (w + 1) * w_wave : M;
        for (int32_t c = c0; c <= c1; ++c)
            for (int32_t s = 0; s < L; ++s)
                m[size_t(landing(s, c, M, L))] |= uint64_t(1) << s;
    };
    std::vector<uint64_t> now(static_cast<size_t>(L)), before(static_cast<size_t>(L));
    written(wave, now);
    written(wave - gens, before);  // the previous wave on the same buffer generation
    for (int32_t j = 0; j < L; ++j)
        zero_mask[j] = before[size_t(j)] & ~now[size_t(j)];
    return TIDE_OK;
}

tide_status_t tide_rs_wave_plan(int32_t M, int32_t L, int32_t w_wave, int32_t k, int32_t me, tide_wave_plan_t *out)
{
    try {
        return rs_wave_plan_impl(M, L, w_wave, k, me, out);
    } catch (...) {
        tide::record_error("host memory allocation failed");
        return TIDE_ERR_OOM;
    }
}

tide_status_t tide_rs_wave_zero_mask(int32_t M, int32_t L, int32_t w_wave, int32_t me, int32_t wave,
                                     uint64_t *zero_mask)
{
    try {
        return rs_wave_zero_mask_impl(M, L, w_wave, me, wave, zero_mask);
    } catch (...) {
        tide::record_error("host memory allocation failed");
        return TIDE_ERR_OOM;
    }
}

int32_t tide_bruck_schedule(int32_t M, int32_t *count, int32_t *step, int32_t max_rounds)
{
    if (M < 1)
        return -1;
    int32_t R = 0;
    while ((int64_t(1) << R) < M)
        ++R;
    if (R > max_rounds || ((!count || !step) && R > 0))
        return -1;
    for (int32_t d = 0; d < R; ++d) {
        step[d] = int32_t(1) << d;
        count[d] = step[d] < M - step[d] ? step[d] : M - step[d];
    }
    return R;
}

}  // extern "C"

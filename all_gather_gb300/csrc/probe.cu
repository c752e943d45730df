// SM-id probe (diagnostic): the measurement behind the TIDE paper's Table 5
// and Figure 3.  Every CTA of the probe records the SM it runs on and its
// entry and exit times (%globaltimer), then holds its SM for a fixed time,
// sized like one wave of a GEMM.  Launched as clusters with a large dynamic
// shared-memory footprint it reproduces a cluster GEMM's placement; probe
// CTAs that enter after the first probe CTA has left were displaced into a
// second wave by whatever else occupied the SMs (here: the reduce-scatter).
// The hold is bounded by time, so the probe always finishes.
#include <cuda_runtime.h>

#include "tide_internal.h"

namespace {

constexpr uint64_t kMaxHoldNs = 10000000ull;  // 10 ms

__device__ __forceinline__ uint64_t now_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One thread that records when the probe's stream reached it: the probe
// CTAs' entry times are measured against it.
__global__ void ready_marker_kernel(uint64_t *t_ready) { *t_ready = now_ns(); }

__global__ void sm_probe_kernel(uint32_t *smid, uint64_t *t_in, uint64_t *t_out, uint64_t hold_ns)
{
    const uint64_t t0 = now_ns();
    if (threadIdx.x == 0) {
        uint32_t id;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
        smid[blockIdx.x] = id;
        t_in[blockIdx.x] = t0;
    }
    while (now_ns() - t0 < hold_ns)
        __nanosleep(200);
    __syncthreads();
    if (threadIdx.x == 0)
        t_out[blockIdx.x] = now_ns();
}

}  // namespace

extern "C" {

tide_status_t tide_sm_probe(int32_t ctas, int32_t cluster, int32_t smem_bytes, uint64_t hold_ns, uint32_t *smid,
                            uint64_t *t_in, uint64_t *t_out, uint64_t *t_ready, void *stream)
{
    tide::record_error("");
    if (ctas < 1 || cluster < 1 || cluster > 8 || ctas % cluster != 0 || smem_bytes < 0 || !smid || !t_in ||
        !t_out || hold_ns > kMaxHoldNs) {
        tide::record_error("need ctas >= 1, 1 <= cluster <= 8 dividing ctas, smem_bytes >= 0, hold_ns <= 10 ms, "
                           "non-NULL outputs");
        return TIDE_ERR_INVALID_ARG;
    }
    cudaError_t e = cudaFuncSetAttribute(sm_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) {
        tide::record_error(cudaGetErrorString(e));
        return TIDE_ERR_CUDA;
    }
    if (t_ready) {
        ready_marker_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(t_ready);
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            tide::record_error(cudaGetErrorString(e));
            return TIDE_ERR_CUDA;
        }
        tide::g_launches.fetch_add(1);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = size_t(smem_bytes);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, sm_probe_kernel, smid, t_in, t_out, hold_ns);
    if (e != cudaSuccess) {
        tide::record_error(cudaGetErrorString(e));
        return TIDE_ERR_CUDA;
    }
    tide::g_launches.fetch_add(1);
    return TIDE_OK;
}

int32_t tide_sm_probe_max_clusters(int32_t cluster, int32_t smem_bytes)
{
    if (cluster < 1 || cluster > 8 || smem_bytes < 0)
        return -1;
    if (cudaFuncSetAttribute(sm_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(cluster));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = size_t(smem_bytes);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sm_probe_kernel, &cfg) != cudaSuccess)
        return -1;
    return n;
}

// Section 2.2, Equation (4): n_gemm GEMM clusters on n_slot - n_blk free
// slots take ceil(n_gemm / (n_slot - n_blk)) waves.  The GEMM keeps one wave
// while the fold blocks at most n_slot - n_gemm slots; a fold CTA that has an
// SM to itself fills one SM of a slot, so that many whole slots hold
// (n_slot - n_gemm) * cluster fold CTAs.
int32_t tide_corun_cta_budget(int32_t cluster_slots, int32_t gemm_ctas, int32_t cluster)
{
    if (cluster_slots < 1 || gemm_ctas < 1 || cluster < 1 || cluster > 16)
        return -1;
    const int64_t n_gemm = (int64_t(gemm_ctas) + cluster - 1) / cluster;
    const int64_t spare = int64_t(cluster_slots) - n_gemm;
    return spare > 0 ? int32_t(spare * cluster) : 0;
}

}  // extern "C"

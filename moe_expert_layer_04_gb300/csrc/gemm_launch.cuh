// gemm_launch.cuh -- host side of the tcgen05 grouped GEMM: tensor maps,
// tile counts, grid size and the launch itself.
#pragma once

#include "gemm_kernel.cuh"

namespace moe {

constexpr int kMaxGroups = 1025;  // E <= 1024 routed experts + the shared one

// max_tiles: an upper bound of the schedule's tiles (CL = 1) or tile pairs
// (CL = 2), used to size the persistent grid.
template <int MODE, int BN, int CL = 1>
moe_status launch_gemm(GemmParams &p, int max_tiles, cudaStream_t st) {
    auto kern = moe_gemm_kernel<MODE, BN, CL>;
    static bool attr_set[64] = {};
    static int max_clusters[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    const int threads = ModeTraits<MODE>::THREADS;
    if (!attr_set[dev]) {
        const int smem_max = (int)gemm_smem_bytes<BN, MODE, CL>(kMaxGroups);
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_max);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        if constexpr (CL == 2) {
            // how many two-CTA clusters can be resident at once
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
            cfg.blockDim = dim3(threads, 1, 1);
            cfg.dynamicSmemBytes = smem_max;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
                return MOE_ERR_CUDA;
            max_clusters[dev] = n;
        }
        attr_set[dev] = true;
    }
    if (max_tiles <= 0) return MOE_OK;
    p.status = device_status_ptr();
    if (!p.status) return MOE_ERR_CUDA;
    if (p.wait_limit <= 0) p.wait_limit = kWaitLimitCycles;
    const size_t smem = gemm_smem_bytes<BN, MODE, CL>(ModeTraits<MODE>::DENSE ? 0 : p.G);
    if constexpr (CL == 1) {
        const int grid = max_tiles < num_sms() ? max_tiles : num_sms();
        kern<<<grid, threads, smem, st>>>(p);
    } else {
        const int clusters = max_tiles < max_clusters[dev] ? max_tiles : max_clusters[dev];
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * clusters, 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return cuda_status(cudaGetLastError());
}


// Upper bound of the 128-row tiles of R rows split into G groups.
inline int row_tile_bound(int max_rows, int G) { return (max_rows + 127) / 128 + G; }

// The same for pairs of 128-row tiles (2-SM MMAs).
inline int row_pair_bound(int max_rows, int G) { return (max_rows + 255) / 256 + G; }

// Which grouped GEMMs may run as 2-SM pairs (bit GM_x; moe_set_gemm_pairs).
int gemm_pair_modes();

// Row-grouped GEMMs pair their tiles when groups hold many row tiles: a
// group with an odd tile count leaves half of its last pair idle.
inline bool rows_pair(int mode, int max_rows, int G) {
    return (gemm_pair_modes() >> mode & 1) && (long long)max_rows >= 1024LL * G;
}

}  // namespace moe

// gemm_launch.cuh -- host side of the tcgen05 grouped GEMM: tensor maps,
// tile counts, grid size and the launch itself.
#pragma once

#include "gemm_kernel.cuh"

namespace moe {

constexpr int kMaxGroups = 1025;  // E <= 1024 routed experts + the shared one

template <int MODE, int BN>
moe_status launch_gemm(GemmParams &p, int max_tiles, cudaStream_t st) {
    auto kern = moe_gemm_kernel<MODE, BN>;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)gemm_smem_bytes<BN, MODE>(kMaxGroups));
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        attr_set[dev] = true;
    }
    if (max_tiles <= 0) return MOE_OK;
    const int grid = max_tiles < num_sms() ? max_tiles : num_sms();
    p.status = device_status_ptr();
    if (!p.status) return MOE_ERR_CUDA;
    if (p.wait_limit <= 0) p.wait_limit = kWaitLimitCycles;
    const size_t smem = gemm_smem_bytes<BN, MODE>(ModeTraits<MODE>::DENSE ? 0 : p.G);
    kern<<<grid, ModeTraits<MODE>::THREADS, smem, st>>>(p);
    return cuda_status(cudaGetLastError());
}

// Upper bound of the 128-row tiles of R rows split into G groups.
inline int row_tile_bound(int max_rows, int G) { return (max_rows + 127) / 128 + G; }

}  // namespace moe

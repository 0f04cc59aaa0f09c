// gemm_bwd.cu -- backward matmuls of the expert FFN (chain rule of the two
// expert matmuls and the clamped SwiGLU of "HyperParallel加速DeepSeek-V4.1
// 多模态1M长序列训练" §2.3 MegaMoE):
//   dgrad 2   dA = dY_perm W2[g]; epilogue: dw = <h, dA>, dH = w dA,
//             dg = dH clamp(u) silu'(min(g,c)) [g <= c], du = dH silu(min(g,c)) [|u| <= c],
//             w h (the wgrad-2 operand)
//   dgrad 1   dX_perm = [dg|du] W13[g]
//   wgrad     dW2[g] = dY_perm_g^T (w h)_g,  dW13[g] = [dg|du]_g^T x_perm_g
//             (contraction over each expert's own rows)
#include <cstring>

#include "gemm_launch.cuh"

namespace moe {

static int dgrad2_bn(int I) { return (I % 256 == 0) ? 256 : (I % 128 == 0) ? 128 : 64; }

// dw partial sums per row: one per column tile and epilogue warp half
int dgrad2_n_tiles(int I) { return I / dgrad2_bn(I) * 2; }

moe_status launch_dgrad2(const uint16_t *dY_perm, const int32_t *offsets, int G, int max_rows,
                         const uint16_t *W2, const float *gu, const float *row_w, int S,
                         int d, int I, float clamp, uint16_t *dGU, uint16_t *hw, float *dw_part,
                         int *dw_tiles, int *tile_counter, cudaStream_t st) {
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    const int BN = dgrad2_bn(I);
    // tiles handed out at run time (see the grouped GEMM): the counter starts at 0
    if (!tile_counter) return MOE_ERR_INVALID_ARG;
    if (cudaMemsetAsync(tile_counter, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    p.tile_counter = tile_counter;
    if (!encode_tmap_bf16_2d(&p.tmA, dY_perm, d, max_rows, (uint64_t)d * 2, 64, 128))
        return MOE_ERR_CUDA;
    // W2 as [G*d rows (contraction), I columns (output)], MN-major boxes
    if (!encode_tmap_bf16_2d(&p.tmB, W2, I, (uint64_t)G * d, (uint64_t)I * 2, 64, 64))
        return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d_sw64(&p.tmO, dGU, 2 * I, max_rows, (uint64_t)4 * I, 32, 32))
        return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d_sw64(&p.tmO2, hw, I, max_rows, (uint64_t)I * 2, 32, 32))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = I / BN;
    p.k_blocks = d / 64;
    p.b_rows_per_group = d;
    p.I = I;
    p.clamp = clamp;
    p.out2 = dGU;
    p.out3 = hw;
    p.out4 = dw_part;
    p.row_w = row_w;
    p.w_rows = S;
    p.gu_in = gu;
    if (dw_tiles) *dw_tiles = dgrad2_n_tiles(I);
    if (BN == 256 && rows_pair(GM_DGRAD2, max_rows, G))
        return launch_gemm<GM_DGRAD2, 256, 2>(p, row_pair_bound(max_rows, G) * p.n_tiles, st);
    const int tiles = row_tile_bound(max_rows, G) * p.n_tiles;
    switch (BN) {
        case 256: return launch_gemm<GM_DGRAD2, 256>(p, tiles, st);
        case 128: return launch_gemm<GM_DGRAD2, 128>(p, tiles, st);
        default: return launch_gemm<GM_DGRAD2, 64>(p, tiles, st);
    }
}

moe_status launch_dgrad1(const uint16_t *dGU, const int32_t *offsets, int G, int max_rows,
                         const uint16_t *W13, int d, int I, uint16_t *dX_perm, cudaStream_t st) {
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    const int BN = (d % 256 == 0) ? 256 : 128;
    if (!encode_tmap_bf16_2d(&p.tmA, dGU, 2 * I, max_rows, (uint64_t)4 * I, 64, 128))
        return MOE_ERR_CUDA;
    // W13 as [G*2I rows (contraction), d columns (output)], MN-major boxes
    if (!encode_tmap_bf16_2d(&p.tmB, W13, d, (uint64_t)G * 2 * I, (uint64_t)d * 2, 64, 64))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = d / BN;
    p.k_blocks = 2 * I / 64;
    p.N = d;
    p.b_rows_per_group = 2 * I;
    p.out = dX_perm;
    if (BN == 256 && rows_pair(GM_DGRAD1, max_rows, G))
        return launch_gemm<GM_DGRAD1, 256, 2>(p, row_pair_bound(max_rows, G) * p.n_tiles, st);
    const int tiles = row_tile_bound(max_rows, G) * p.n_tiles;
    return BN == 256 ? launch_gemm<GM_DGRAD1, 256>(p, tiles, st)
                     : launch_gemm<GM_DGRAD1, 128>(p, tiles, st);
}

// One CTA, a thread per group (G <= 1025):
//   maps[g]    a copy of A's tensor map whose rows end at the group's last
//              row; the weight-gradient producer loads a group's ragged last
//              k-block through it, so that the rows past the group land as
//              zeros;
//   korder[r]  the group of rank r in order of decreasing rows (ties by
//              index): the schedule takes the long contractions first;
//   *counter   0, the tiles the GEMM has handed out.
__global__ void __launch_bounds__(1024) wgrad_prep_kernel(const __grid_constant__ CUtensorMap tmpl,
                                                         const int32_t *offsets, int G,
                                                         CUtensorMap *maps, int32_t *korder,
                                                         int *counter) {
    __shared__ int32_t rows_s[1025];
    if (threadIdx.x == 0) *counter = 0;
    for (int g = threadIdx.x; g < G; g += blockDim.x) rows_s[g] = offsets[g + 1] - offsets[g];
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(&tmpl);
        uint4 *dst = reinterpret_cast<uint4 *>(maps + g);
#pragma unroll
        for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) dst[i] = src[i];
        const int end = offsets[g + 1];
        tmap_replace_dim1(maps + g, (uint32_t)(end > 0 ? end : 1));
        const int rg = rows_s[g];
        int rank = 0;
        for (int h = 0; h < G; ++h) {
            const int rh = rows_s[h];
            rank += (rh > rg || (rh == rg && h < g)) ? 1 : 0;
        }
        korder[rank] = g;
    }
    fence_tmap_release();
}

moe_status launch_wgrad(const uint16_t *A, int M, const uint16_t *B, int N, const int32_t *offsets,
                        int G, int R, float *dW, void *scratch, cudaStream_t st) {
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    if (M % 128 != 0 || N % 64 != 0) return MOE_ERR_UNSUPPORTED;
    static_assert(sizeof(CUtensorMap) == 128, "tensor maps of 128 bytes");
    if (G < 1 || G > 1025 || !scratch || (reinterpret_cast<uintptr_t>(scratch) & 63u) != 0)
        return MOE_ERR_INVALID_ARG;
    // Short contractions (few rows per group) make the fp32 output stream the
    // bound: 128-wide tiles keep more operand stages in flight.  Long ones are
    // tensor-bound: 256-wide tiles halve the operand reads per FLOP.
    const bool long_k = (long long)R >= 512LL * G;
    const int BN = (long_k && N % 256 == 0) ? 256 : (N % 128 == 0) ? 128 : 64;
    if (!encode_tmap_bf16_2d(&p.tmA, A, M, R, (uint64_t)M * 2, 64, 64)) return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d(&p.tmB, B, N, R, (uint64_t)N * 2, 64, 64)) return MOE_ERR_CUDA;
    CUtensorMap *maps = static_cast<CUtensorMap *>(scratch);
    int32_t *korder = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(scratch) +
                                                  (size_t)1025 * sizeof(CUtensorMap));
    int *counter = scratch_tile_counter(scratch);
    wgrad_prep_kernel<<<1, 1024, 0, st>>>(p.tmA, offsets, G, maps, korder, counter);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    p.tail_maps = maps;
    p.korder = korder;
    p.tile_counter = counter;
    p.offsets = offsets;
    p.G = G;
    p.m_tiles = M / 128;
    p.n_tiles = N / BN;
    p.N = N;
    p.M = M;
    p.out = dW;
    const int tiles = G * p.m_tiles * p.n_tiles;
    // long contractions: 2-SM pairs, two 128-row output tiles sharing one B
    // tile, each CTA loading half of it
    if (BN == 256 && p.m_tiles % 2 == 0 && (gemm_pair_modes() >> GM_WGRAD & 1))
        return launch_gemm<GM_WGRAD, 256, 2>(p, tiles / 2, st);
    switch (BN) {
        case 256: return launch_gemm<GM_WGRAD, 256>(p, tiles, st);
        case 128: return launch_gemm<GM_WGRAD, 128>(p, tiles, st);
        default: return launch_gemm<GM_WGRAD, 64>(p, tiles, st);
    }
}

}  // namespace moe

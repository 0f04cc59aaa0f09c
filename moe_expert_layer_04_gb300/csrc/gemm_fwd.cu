// gemm_fwd.cu -- forward matmuls: gate projection and the two expert GEMMs.
//
//   gate projection  logits = x W_g^T (+ offset)   ("HyperParallel加速DeepSeek-V4.1
//                    多模态1M长序列训练" §2.3, MegaGate: the projection stays an
//                    ordinary matmul ahead of the routing pipeline)
//   expert GEMM 1    [g|u] = x_perm W13[g]^T, h = silu(min(g,c)) clamp(u,-c,c)
//   expert GEMM 2    y = w * (h W2[g]^T)          (same page, §2.3 MegaMoE: two
//                    expert matmuls around SwiGLU with the V4.1 clamp)
#include <cstring>

#include "gemm_launch.cuh"

namespace moe {

template <int BN>
static moe_status gate_gemm_bn(const uint16_t *x, const uint16_t *Wg, const float *offset, int T,
                               int d, int E, float *logits, cudaStream_t st) {
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    if (!encode_tmap_bf16_2d(&p.tmA, x, d, T, (uint64_t)d * 2, 64, 128)) return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d(&p.tmB, Wg, d, E, (uint64_t)d * 2, 64, BN)) return MOE_ERR_CUDA;
    p.G = 1;
    p.rows = T;
    p.n_tiles = (E + BN - 1) / BN;
    p.k_blocks = d / 64;
    p.N = E;
    p.out = logits;
    p.col_add = offset;
    return launch_gemm<GM_GATE, BN>(p, ((T + 127) / 128) * p.n_tiles, st);
}

moe_status launch_gate_gemm(const uint16_t *x, const uint16_t *Wg, const float *offset, int T,
                            int d, int E, float *logits, cudaStream_t st) {
    // 128-wide tiles read each x tile half as often; use them when they still
    // give every SM at least two tiles
    const long long tiles128 = (long long)((T + 127) / 128) * ((E + 127) / 128);
    if (tiles128 >= 2LL * num_sms())
        return gate_gemm_bn<128>(x, Wg, offset, T, d, E, logits, st);
    return gate_gemm_bn<64>(x, Wg, offset, T, d, E, logits, st);
}

moe_status launch_ffn1(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                       const uint16_t *W13, int d, int I, float clamp, uint16_t *h,
                       float *gu_save, cudaStream_t st) {
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    const int BN = (I % 128 == 0) ? 256 : 128;
    if (!encode_tmap_bf16_2d(&p.tmA, x_perm, d, max_rows, (uint64_t)d * 2, 64, 128))
        return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d(&p.tmB, W13, d, (uint64_t)G * 2 * I, (uint64_t)d * 2, 64, BN / 2))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = I / (BN / 2);
    p.k_blocks = d / 64;
    p.b_rows_per_group = 2 * I;
    p.I = I;
    p.clamp = clamp;
    p.out = h;
    p.out2 = gu_save;
    if (BN == 256 && rows_pair(GM_FFN1, max_rows, G))
        return launch_gemm<GM_FFN1, 256, 2>(p, row_pair_bound(max_rows, G) * p.n_tiles, st);
    const int tiles = row_tile_bound(max_rows, G) * p.n_tiles;
    return BN == 256 ? launch_gemm<GM_FFN1, 256>(p, tiles, st)
                     : launch_gemm<GM_FFN1, 128>(p, tiles, st);
}

moe_status launch_ffn2(const uint16_t *h, const int32_t *offsets, int G, int max_rows,
                       const uint16_t *W2, const float *row_w, int S, int d, int I, uint16_t *y,
                       cudaStream_t st) {
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    const int BN = (d % 256 == 0) ? 256 : 128;
    const bool pair = BN == 256 && rows_pair(GM_FFN2, max_rows, G);
    if (!encode_tmap_bf16_2d(&p.tmA, h, I, max_rows, (uint64_t)I * 2, 64, 128))
        return MOE_ERR_CUDA;
    // a pair's CTAs each load half of the B tile's rows
    if (!encode_tmap_bf16_2d(&p.tmB, W2, I, (uint64_t)G * d, (uint64_t)I * 2, 64,
                             pair ? BN / 2 : BN))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = d / BN;
    p.k_blocks = I / 64;
    p.N = d;
    p.b_rows_per_group = d;
    p.out = y;
    p.row_w = row_w;
    p.w_rows = S;
    if (pair) return launch_gemm<GM_FFN2, 256, 2>(p, row_pair_bound(max_rows, G) * p.n_tiles, st);
    const int tiles = row_tile_bound(max_rows, G) * p.n_tiles;
    return BN == 256 ? launch_gemm<GM_FFN2, 256>(p, tiles, st)
                     : launch_gemm<GM_FFN2, 128>(p, tiles, st);
}

}  // namespace moe

namespace moe {

// One readiness counter per 128-row tile of the grouped row space.
int ffn_fused_counters(int max_rows, int G) { return row_tile_bound(max_rows, G); }

moe_status launch_ffn12(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                        const uint16_t *W13, const uint16_t *W2, const float *row_w, int S, int d,
                        int I, float clamp, uint16_t *h, float *gu_save, uint16_t *y, int *ready,
                        cudaStream_t st, int stall_rt, long long wait_limit) {
    if (I % 128 != 0 || d % 256 != 0) return MOE_ERR_UNSUPPORTED;
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    constexpr int BN = 256;
    // GEMM 1: [g|u] = x_perm W13[g]^T, 128 h columns (gate and up halves) per tile
    if (!encode_tmap_bf16_2d(&p.tmA, x_perm, d, max_rows, (uint64_t)d * 2, 64, 128))
        return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d(&p.tmB, W13, d, (uint64_t)G * 2 * I, (uint64_t)d * 2, 64, BN / 2))
        return MOE_ERR_CUDA;
    // GEMM 2: y = w (h W2[g]^T), 256 output columns per tile
    if (!encode_tmap_bf16_2d(&p.tmO, h, I, max_rows, (uint64_t)I * 2, 64, 128))
        return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d(&p.tmO2, W2, I, (uint64_t)G * d, (uint64_t)I * 2, 64, BN))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = I / (BN / 2);
    p.k_blocks = d / 64;
    p.b_rows_per_group = 2 * I;
    p.I = I;
    p.clamp = clamp;
    p.out = h;
    p.out2 = gu_save;
    p.out3 = y;
    p.N = d;
    p.n_tiles2 = d / BN;
    p.k_blocks2 = I / 64;
    p.b_rows2 = d;
    p.row_w = row_w;
    p.w_rows = S;
    p.ready = ready;
    p.ready_target = p.n_tiles * ModeTraits<GM_FFN12>::NEPI;
    p.stall_rt = stall_rt;
    p.wait_limit = wait_limit;
    const int rt = ffn_fused_counters(max_rows, G);
    if (cudaMemsetAsync(ready, 0, (size_t)rt * sizeof(int), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_gemm<GM_FFN12, BN>(p, rt * (p.n_tiles + p.n_tiles2), st);
}

}  // namespace moe

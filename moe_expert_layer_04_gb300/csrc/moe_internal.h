// moe_internal.h -- declarations shared by the translation units of libmoe.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// Default limit of every bounded device-side wait, in SM clock cycles
// (about four seconds at 2 GHz; the longest legitimate wait is one tile).
constexpr long long kWaitLimitCycles = 1LL << 33;

// Address of this library's status word on the current device.
int *device_status_ptr();

// Number of SMs of the current device (cached per device).
int num_sms();

// Encodes a 2-D bf16 tensor map with 128-byte swizzle: a [outer, inner]
// row-major matrix with the given row pitch (bytes), copied in boxes of
// box_inner x box_outer elements.  Out-of-bounds elements read as zero.
bool encode_tmap_bf16_2d(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                         uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer);

// bf16 2-D matrix with 64-byte swizzle (boxes with a 64-byte inner extent).
bool encode_tmap_bf16_2d_sw64(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                              uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer);

// Same for a 2-D fp32 matrix (stores), 128-byte swizzle.
bool encode_tmap_f32_2d(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                        uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer);

// 2-D byte matrix (MXFP8 codes or scale codes); swizzle_bytes 128, 64 or 0
// (none).
bool encode_tmap_u8_2d(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                       uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer,
                       int swizzle_bytes);

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Supported-shape check shared by the entry points.
moe_status check_shapes(int T, int d, int E, int k, int I);

// ------------------------------------------------------------ kernels

// Grouped / dense GEMM modes of the tcgen05 kernel.
enum GemmMode : int {
    GM_GATE = 0,    // logits = x W_g^T (+ offset), fp32 out
    GM_FFN1 = 1,    // [g|u] = x_perm W13[g]^T -> clamped SwiGLU h (bf16), optional g|u save
    GM_FFN2 = 2,    // y = w * (h W2[g]^T) (bf16)
    GM_DGRAD2 = 3,  // dA = dY_perm W2[g] -> clamped-SwiGLU backward (dGU, w h, dw partials)
    GM_DGRAD1 = 4,  // dX_perm = dGU W13[g] (bf16)
    GM_WGRAD = 5,   // dW[g] = A_g^T B_g over the group's rows (fp32)
    GM_FFN12 = 6    // GM_FFN1 then GM_FFN2 in one persistent launch, each GEMM-2 row
                    // tile waiting for the GEMM-1 tiles that produce its h rows
};

// Host launchers (gemm_*.cu).  All pointers are device pointers.
moe_status launch_gate_gemm(const uint16_t *x, const uint16_t *Wg, const float *offset, int T,
                            int d, int E, float *logits, cudaStream_t st);
moe_status launch_ffn1(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                       const uint16_t *W13, int d, int I, float clamp, uint16_t *h,
                       float *gu_save, cudaStream_t st);
// Both expert GEMMs in one launch (needs I % 128 == 0 and d % 256 == 0);
// `ready` holds ffn_fused_counters(max_rows, G) ints of the caller's workspace.
int ffn_fused_counters(int max_rows, int G);
moe_status launch_ffn12(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                        const uint16_t *W13, const uint16_t *W2, const float *row_w, int S, int d,
                        int I, float clamp, uint16_t *h, float *gu_save, uint16_t *y, int *ready,
                        cudaStream_t st, int stall_rt = -1, long long wait_limit = 0);
moe_status launch_ffn2(const uint16_t *h, const int32_t *offsets, int G, int max_rows,
                       const uint16_t *W2, const float *row_w, int S, int d, int I, uint16_t *y,
                       cudaStream_t st);
moe_status launch_dgrad2(const uint16_t *dY_perm, const int32_t *offsets, int G, int max_rows,
                         const uint16_t *W2, const float *gu, const float *row_w, int S,
                         int d, int I, float clamp, uint16_t *dGU, uint16_t *hw, float *dw_part,
                         int *dw_tiles, int *tile_counter, cudaStream_t st);
int dgrad2_n_tiles(int I);
moe_status launch_dgrad1(const uint16_t *dGU, const int32_t *offsets, int G, int max_rows,
                         const uint16_t *W13, int d, int I, uint16_t *dX_perm, cudaStream_t st);
// dW[g] (M x N, fp32) = A[rows of g]^T B[rows of g]; A [R, M] and B [R, N] bf16.
// scratch: kWgradScratchBytes of device memory (64-byte aligned) for the
// per-group tensor maps of A, the schedule's group order and its tile
// counter; calls in order on one stream may share it.
constexpr size_t kWgradScratchBytes = (size_t)1025 * 128 + (size_t)1025 * 4 + 64;
// The tile counter inside that scratch (also dgrad 2's, which runs first).
inline int *scratch_tile_counter(void *scratch) {
    return reinterpret_cast<int *>(static_cast<uint8_t *>(scratch) + (size_t)1025 * 128 +
                                   (size_t)1025 * 4);
}
moe_status launch_wgrad(const uint16_t *A, int M, const uint16_t *B, int N, const int32_t *offsets,
                        int G, int R, float *dW, void *scratch, cudaStream_t st);

// Row gather: dst[row] = src[row_token[row]] for the S routed rows plus the
// T identity rows, reading each token row once (permute.cu).
moe_status launch_gather_rows(const uint16_t *src, const int32_t *slot_row, int T, int d, int k,
                              uint16_t *dst, cudaStream_t st);

// MXFP8 (mx.cu, gemm_mx.cu): quantisation of bf16 rows (along the rows of a
// stack of matrices, written transposed: src [G, R, C] -> q [G*C, R]), the
// quantising dispatch gather, the two MX expert GEMMs and the MX dgrad 2
// (d % 256 == 0, I % 128 == 0); MX dgrad 1 is launch_mx_ffn2 with K = 2I.
moe_status launch_mx_quantize(const uint16_t *src, long long rows, int K, uint8_t *q, uint8_t *sf,
                              cudaStream_t st);
moe_status launch_mx_quantize_t(const uint16_t *src, int G, int R, int C, uint8_t *q, uint8_t *sf,
                                cudaStream_t st);
moe_status launch_mx_quantize_both(const uint16_t *src, int G, int R, int C, uint8_t *q,
                                   uint8_t *sf, uint8_t *qt, uint8_t *sft, cudaStream_t st);
moe_status launch_mx_gather(const uint16_t *x, const int32_t *slot_row, int T, int d, int k,
                            uint8_t *q, uint8_t *sf, cudaStream_t st);
moe_status launch_mx_ffn1(const uint8_t *xq, const uint8_t *xsf, const int32_t *offsets, int G,
                          int max_rows, const uint8_t *W13q, const uint8_t *W13sf, int d, int I,
                          float clamp, uint8_t *hq, uint8_t *hsf, float *gu_save,
                          cudaStream_t st);
moe_status launch_mx_ffn2(const uint8_t *hq, const uint8_t *hsf, const int32_t *offsets, int G,
                          int max_rows, const uint8_t *W2q, const uint8_t *W2sf,
                          const float *row_w, int S, int d, int I, uint16_t *y, cudaStream_t st);
// MX weight gradients: the padded contraction plan (kofs, sofs [G+1]), the
// quantisation of each group's rows along the rows, written transposed in
// the K-chunk-major layout (codes of (c, k) at ((k/128) C + c) 128 + k%128,
// scale codes in 16-byte slots likewise; row r read from src[row_idx[r]]
// when row_idx is given), and dW[g] (M x N fp32) over group g's padded
// contraction of At (C = M) and Bt (C = N) in that layout; k_chunks and
// sf_slots bound the chunks of 128 codes and the 16-byte scale slots.
moe_status launch_mx_kpad_plan(const int32_t *offsets, int G, int32_t *kofs, int32_t *sofs,
                               cudaStream_t st);
moe_status launch_mx_quantize_rows_t(const uint16_t *src, const int32_t *row_idx,
                                     const int32_t *offsets, const int32_t *kofs,
                                     const int32_t *sofs, int G, int max_tiles, int C,
                                     uint8_t *qt, uint8_t *sft, cudaStream_t st);
moe_status launch_mx_wgrad(const uint8_t *At, const uint8_t *Atsf, const uint8_t *Bt,
                           const uint8_t *Btsf, const int32_t *kofs, const int32_t *sofs, int G,
                           int M, int N, int k_chunks, int sf_slots, float *dW, int32_t *korder,
                           int *tile_counter, cudaStream_t st);
// Partials of <h~, dA> per row written by launch_mx_dgrad2.
int mx_dgrad2_n_part(int I);
moe_status launch_mx_dgrad2(const uint8_t *dYq, const uint8_t *dYsf, const int32_t *offsets, int G,
                            int max_rows, const uint8_t *W2tq, const uint8_t *W2tsf,
                            const float *gu, const uint8_t *hq, const uint8_t *hsf,
                            const float *row_w, int S, int d, int I, float clamp, uint16_t *dGU,
                            uint8_t *dGUq, uint8_t *dGUsf, uint16_t *hw, float *dw_part,
                            int *n_part, int *tile_counter, cudaStream_t st);

moe_status launch_selftest_timeout(long long limit, cudaStream_t st);

// Row movement around an exchange between GPUs (exchange.cu).
moe_status launch_index_gather(const void *src, const int32_t *idx, long long n, long long n_src,
                               int row_bytes, void *dst, cudaStream_t st);
moe_status launch_row_sum(const float *part, long long n, int n_part, float *out,
                          cudaStream_t st);

}  // namespace moe

namespace moe {
// the MOE_PAIR_* bits of moe.h are the GemmMode values
static_assert(MOE_PAIR_EXPERT_GEMM1 == 1 << GM_FFN1 && MOE_PAIR_EXPERT_GEMM2 == 1 << GM_FFN2 &&
                  MOE_PAIR_DGRAD2 == 1 << GM_DGRAD2 && MOE_PAIR_DGRAD1 == 1 << GM_DGRAD1 &&
                  MOE_PAIR_WGRAD == 1 << GM_WGRAD,
              "pair bits follow the matmul modes");
}  // namespace moe

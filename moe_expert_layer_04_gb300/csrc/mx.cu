// mx.cu -- MXFP8 quantisation of bf16 matrices along their rows, and the
// dispatch gather that quantises each token row once and writes it to the
// token's k routed rows and to its shared-expert row.
//
// Layout of a quantised [rows, K] matrix: codes q [rows, K] (one E4M3 code
// per byte, row-major) and scales sf [rows, mx_sf_pitch(K)] (the E8M0 code of
// block b of row r at sf[r * pitch + b]; the padding bytes are not written).
#include "moe_internal.h"
#include "mx_common.cuh"

namespace moe {
namespace {

// 32 bf16 values (64 bytes, 16-byte aligned) -> fp32 (exact).
__device__ __forceinline__ void load_block_bf16(const uint16_t *p, float (&v)[32]) {
    const uint4 *s = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 u = __ldg(s + j);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[8 * j + 2 * e] = __uint_as_float(w[e] << 16);
            v[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
    }
}

__device__ __forceinline__ void store_block(uint8_t *q, const uint32_t (&w)[8]) {
    uint4 *d = reinterpret_cast<uint4 *>(q);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// One thread per block of 32; consecutive threads take consecutive blocks of
// a row, so a warp reads 2 KB and writes 1 KB of codes contiguously.
__global__ void __launch_bounds__(256)
    mx_quantize_kernel(const uint16_t *__restrict__ src, long long nblk, int kb32, int K, int sfp,
                       uint8_t *__restrict__ q, uint8_t *__restrict__ sf) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nblk; i += stride) {
        const long long r = i / kb32;
        const int b = (int)(i - r * kb32);
        float v[32];
        load_block_bf16(src + (size_t)r * K + (size_t)b * 32, v);
        uint32_t w[8];
        const uint32_t code = mx_quantize_block(v, w);
        store_block(q + (size_t)r * K + (size_t)b * 32, w);
        sf[(size_t)r * sfp + b] = (uint8_t)code;
    }
}

// One warp per token; lanes take the row's blocks, kU per lane per pass.
constexpr int kU = 2;

__global__ void __launch_bounds__(256)
    mx_gather_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ slot_row, int T,
                     int d, int k, int sfp, uint8_t *__restrict__ q, uint8_t *__restrict__ sf) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nw = gridDim.x * 8;
    const size_t S = (size_t)T * k;
    const int nb = d / 32;
    for (int t = gw; t < T; t += nw) {
        int row = 0;
        if (lane < k) row = slot_row[(size_t)t * k + lane];
        // every lane runs the same iterations: the shuffles below need the full warp
        for (int b0 = 0; b0 < nb; b0 += 32 * kU) {
            uint32_t w[kU][8];
            uint32_t code[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int b = b0 + lane + 32 * u;
                if (b < nb) {
                    float v[32];
                    load_block_bf16(x + (size_t)t * d + (size_t)b * 32, v);
                    code[u] = mx_quantize_block(v, w[u]);
                }
            }
            for (int j = 0; j <= k; ++j) {
                const size_t r = j < k ? (size_t)__shfl_sync(0xffffffffu, row, j) : S + t;
                if (j < k && r >= S) continue;     // not a routed row (invalid dispatch)
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int b = b0 + lane + 32 * u;
                    if (b < nb) {
                        store_block(q + r * d + (size_t)b * 32, w[u]);
                        sf[r * sfp + b] = (uint8_t)code[u];
                    }
                }
            }
        }
    }
}

// Quantisation along the rows of a stack of matrices, written transposed:
// for src [G, R, C] bf16, output row g*C + c is column c of matrix g (R
// values) quantised in blocks of 32 along R.  One thread per output block;
// consecutive threads take consecutive columns, so each of the 32 loads of a
// warp reads 64 contiguous bytes.
__global__ void __launch_bounds__(256)
    mx_quantize_t_kernel(const uint16_t *__restrict__ src, int G, int R, int C, int sfp,
                         uint8_t *__restrict__ q, uint8_t *__restrict__ sf) {
    const long long nb = (long long)G * (R / 32) * C;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nb; i += stride) {
        const int c = (int)(i % C);
        const long long gb = i / C;
        const int b = (int)(gb % (R / 32));
        const int g = (int)(gb / (R / 32));
        const uint16_t *col = src + ((size_t)g * R + (size_t)b * 32) * C + c;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float((uint32_t)__ldg(col + (size_t)j * C) << 16);
        uint32_t w[8];
        const uint32_t code = mx_quantize_block(v, w);
        const size_t orow = (size_t)g * C + c;
        store_block(q + orow * R + (size_t)b * 32, w);
        sf[orow * sfp + b] = (uint8_t)code;
    }
}

}  // namespace

moe_status launch_mx_quantize_t(const uint16_t *src, int G, int R, int C, uint8_t *q, uint8_t *sf,
                                cudaStream_t st) {
    const long long nb = (long long)G * (R / 32) * C;
    if (nb == 0) return MOE_OK;
    const long long want = (nb + 255) / 256;
    const int blocks = (int)(want < (long long)num_sms() * 16 ? want : (long long)num_sms() * 16);
    mx_quantize_t_kernel<<<blocks, 256, 0, st>>>(src, G, R, C, mx_sf_pitch(R), q, sf);
    return cuda_status(cudaGetLastError());
}

moe_status launch_mx_quantize(const uint16_t *src, long long rows, int K, uint8_t *q, uint8_t *sf,
                              cudaStream_t st) {
    const long long nblk = rows * (K / 32);
    if (nblk == 0) return MOE_OK;
    const long long want = (nblk + 255) / 256;
    const int blocks = (int)(want < (long long)num_sms() * 16 ? want : (long long)num_sms() * 16);
    mx_quantize_kernel<<<blocks, 256, 0, st>>>(src, nblk, K / 32, K, mx_sf_pitch(K), q, sf);
    return cuda_status(cudaGetLastError());
}

moe_status launch_mx_gather(const uint16_t *x, const int32_t *slot_row, int T, int d, int k,
                            uint8_t *q, uint8_t *sf, cudaStream_t st) {
    const int want = (T + 7) / 8;
    const int blocks = want < num_sms() * 8 ? want : num_sms() * 8;
    mx_gather_kernel<<<blocks, 256, 0, st>>>(x, slot_row, T, d, k, mx_sf_pitch(d), q, sf);
    return cuda_status(cudaGetLastError());
}

}  // namespace moe

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

// Both orientations of a stack of matrices in one pass: for src [G, R, C]
// bf16 (R, C multiples of 128), q [G*R, C] quantised along C (rows) and qt
// [G*C, R] quantised along R (columns, written transposed).  A CTA takes
// 128 x 128 tiles: its 256 threads stage the tile in shared memory, then
// threads 0-127 quantise one row each (4 blocks) while threads 128-255
// quantise one column each (4 blocks along R); both write their codes to
// staging tiles in shared memory and their four scale codes as one 32-bit
// word, and all threads then copy the two code tiles out with coalesced
// 16-byte stores (eight threads per 128-byte row).  Row pitches padded by
// 16 bytes keep every shared-memory pass free of bank conflicts.  The next
// tile's loads are in flight during the quantisation.
constexpr int kQT = 128;                  // tile edge
constexpr int kQTPitch = kQT * 2 + 16;    // bytes per staged bf16 row
constexpr int kQCPitch = kQT + 16;        // bytes per staged code row
constexpr int kQSmem = kQT * kQTPitch + 2 * kQT * kQCPitch;

__global__ void __launch_bounds__(256)
    mx_quantize_both_kernel(const uint16_t *__restrict__ src, int G, int R, int C, int sfpC,
                            int sfpR, uint8_t *__restrict__ q, uint8_t *__restrict__ sf,
                            uint8_t *__restrict__ qt, uint8_t *__restrict__ sft) {
    extern __shared__ __align__(16) uint8_t qsm[];
    uint8_t *tile = qsm;                              // [128][kQTPitch] bf16 rows
    uint8_t *cq = qsm + kQT * kQTPitch;               // [128 rows][kQCPitch] codes along C
    uint8_t *cqt = cq + kQT * kQCPitch;               // [128 cols][kQCPitch] codes along R
    const int tr = R / kQT, tc = C / kQT;
    const long long n_tiles = (long long)G * tr * tc;
    const int t = threadIdx.x;
    // column tiles fastest: the scale words of a row fill their 32-byte
    // sectors within a few consecutive tiles
    auto origin = [&](long long i, int &g, int &r0, int &c0) {
        c0 = (int)(i % tc) * kQT;
        const long long rest = i / tc;
        r0 = (int)(rest % tr) * kQT;
        g = (int)(rest / tr);
    };
    // the tile's 16-byte chunks of this thread (16 per row), loaded into
    // registers one tile ahead
    uint4 v[8];
    auto load = [&](long long i) {
        int g, r0, c0;
        origin(i, g, r0, c0);
        const uint16_t *base = src + ((size_t)g * R + r0) * C + c0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int chunk = t + 256 * j;
            v[j] = __ldg(reinterpret_cast<const uint4 *>(base + (size_t)(chunk >> 4) * C) +
                         (chunk & 15));
        }
    };
    if ((long long)blockIdx.x < n_tiles) load(blockIdx.x);
    for (long long i = blockIdx.x; i < n_tiles; i += gridDim.x) {
        int g, r0, c0;
        origin(i, g, r0, c0);
        __syncthreads();   // the previous tile's readers and copiers are done
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int chunk = t + 256 * j;
            *reinterpret_cast<uint4 *>(tile + (chunk >> 4) * kQTPitch + (chunk & 15) * 16) = v[j];
        }
        __syncthreads();
        if (i + gridDim.x < n_tiles) load(i + gridDim.x);
        uint32_t codes = 0;
        if (t < kQT) {
            // row r0 + t: four blocks along C
            const uint8_t *rowp = tile + t * kQTPitch;
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
                float f[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(rowp + b * 64 + j * 16);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        f[8 * j + 2 * e] = __uint_as_float(w[e] << 16);
                        f[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                    }
                }
                uint32_t w[8];
                codes |= mx_quantize_block(f, w) << (8 * b);
                store_block(cq + t * kQCPitch + b * 32, w);
            }
            *reinterpret_cast<uint32_t *>(sf + ((size_t)g * R + r0 + t) * sfpC + c0 / 32) = codes;
        } else {
            // column c0 + (t - 128): four blocks along R
            const int c = t - kQT;
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    f[j] = __uint_as_float(
                        (uint32_t)*reinterpret_cast<const uint16_t *>(tile + (b * 32 + j) * kQTPitch +
                                                                      c * 2)
                        << 16);
                uint32_t w[8];
                codes |= mx_quantize_block(f, w) << (8 * b);
                store_block(cqt + c * kQCPitch + b * 32, w);
            }
            *reinterpret_cast<uint32_t *>(sft + ((size_t)g * C + c0 + c) * sfpR + r0 / 32) = codes;
        }
        __syncthreads();
        // both code tiles out: 8 chunks of 16 bytes per 128-byte row
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int chunk = t + 256 * j;
            const int row = chunk >> 3, c16 = (chunk & 7) * 16;
            *reinterpret_cast<uint4 *>(q + ((size_t)g * R + r0 + row) * C + c0 + c16) =
                *reinterpret_cast<const uint4 *>(cq + row * kQCPitch + c16);
            *reinterpret_cast<uint4 *>(qt + ((size_t)g * C + c0 + row) * R + r0 + c16) =
                *reinterpret_cast<const uint4 *>(cqt + row * kQCPitch + c16);
        }
    }
}

// The padded contraction of the MX weight gradients: group g's rows occupy
// kpad_g = cnt_g rounded up to 128 columns of the transposed operands,
// starting at kofs[g]; its scale codes kpad_g / 32 bytes starting at
// sofs[g], a multiple of 16 (16-byte TMA rows).  One warp, a scan over the
// groups in chunks of 32.
__global__ void mx_kpad_plan_kernel(const int32_t *__restrict__ offsets, int G,
                                    int32_t *__restrict__ kofs, int32_t *__restrict__ sofs) {
    const int lane = threadIdx.x & 31;
    int kc = 0, sc = 0;
    for (int base = 0; base <= G; base += 32) {
        const int g = base + lane;
        int kp = 0, sp = 0;
        if (g < G) {
            const int cnt = offsets[g + 1] - offsets[g];
            kp = (cnt + 127) / 128 * 128;
            sp = (kp / 32 + 15) / 16 * 16;
        }
        int ki = kp, si = sp;
#pragma unroll
        for (int sft = 1; sft < 32; sft <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, ki, sft);
            const int b = __shfl_up_sync(0xffffffffu, si, sft);
            if (lane >= sft) { ki += a; si += b; }
        }
        if (g <= G) {
            kofs[g] = kc + ki - kp;
            sofs[g] = sc + si - sp;
        }
        kc += __shfl_sync(0xffffffffu, ki, 31);
        sc += __shfl_sync(0xffffffffu, si, 31);
    }
}

// Quantisation along the rows of each group, written transposed: for the
// permuted rows src [R, C] bf16 (row r read from src row row_idx[r] when
// row_idx is given), column c of group g's rows, in blocks of 32 rows from
// the group's first row (the last block zero-padded).  The transposed
// operand is K-chunk-major, so that each stage of the weight-gradient GEMM
// reads one contiguous box: code (c, k) of the padded contraction
// k in [kofs[g], kofs[g] + kpad_g) at qt[((k / 128) * C + c) * 128 + k % 128];
// scale code (c, j) of the group's j-th block at
// sft[((sofs[g] / 16 + j / 16) * C + c) * 16 + j % 16].  A CTA takes 128 x 128
// tiles (128 padded rows of one group, 128 columns): its 256 threads stage
// the tile in shared memory (rows past the group's end as zeros), each
// thread quantises two 32-row blocks of one column into a staging tile of
// codes, and all threads copy the codes out with coalesced 16-byte stores.
__global__ void __launch_bounds__(256, 3)
    mx_quantize_rows_t_kernel(const uint16_t *__restrict__ src, const int32_t *__restrict__ row_idx,
                              const int32_t *__restrict__ offsets,
                              const int32_t *__restrict__ kofs, const int32_t *__restrict__ sofs,
                              int G, int C, uint8_t *__restrict__ qt, uint8_t *__restrict__ sft) {
    extern __shared__ __align__(16) uint8_t qsm[];
    uint8_t *tile = qsm;                         // [128 rows][kQTPitch] bf16
    uint8_t *cqt = qsm + kQT * kQTPitch;         // [128 columns][kQCPitch] codes
    // per group: first row tile, first row, first scale slot ([G+1] each)
    int *s_tile0 = reinterpret_cast<int *>(cqt + kQT * kQCPitch);
    int *s_row0 = s_tile0 + (G + 1);
    int *s_slot0 = s_row0 + (G + 1);
    const int t = threadIdx.x;
    for (int g = t; g <= G; g += blockDim.x) {
        s_tile0[g] = kofs[g] / kQT;
        s_row0[g] = offsets[g];
        s_slot0[g] = sofs[g] / 16;
    }
    __syncthreads();
    const int tc = C / kQT;
    const long long n_tiles = (long long)s_tile0[G] * tc;
    struct Tile {
        int g, rt, r0, valid, c0;
    };
    auto locate = [&](long long i) {
        Tile tl;
        const int rtg = (int)(i / tc);          // row tile over all groups
        int lo = 0, hi = G - 1;                 // the group holding it
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_tile0[mid] <= rtg) lo = mid; else hi = mid - 1;
        }
        tl.g = lo;
        tl.rt = rtg - s_tile0[lo];
        tl.r0 = s_row0[lo] + tl.rt * kQT;
        tl.valid = min(kQT, s_row0[lo + 1] - tl.r0);
        tl.c0 = (int)(i % tc) * kQT;
        return tl;
    };
    // the tile's 16-byte chunks of this thread (16 per row; rows past the
    // group's end are zeros), loaded into registers one tile ahead
    uint4 v[8];
    auto load = [&](const Tile &tl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int chunk = t + 256 * j;
            const int r = chunk >> 4;
            v[j] = make_uint4(0u, 0u, 0u, 0u);
            if (r < tl.valid) {
                const int sr = row_idx ? row_idx[tl.r0 + r] : tl.r0 + r;
                v[j] = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)sr * C + tl.c0) +
                             (chunk & 15));
            }
        }
    };
    Tile cur{};
    if ((long long)blockIdx.x < n_tiles) {
        cur = locate(blockIdx.x);
        load(cur);
    }
    for (long long i = blockIdx.x; i < n_tiles; i += gridDim.x) {
        const Tile tl = cur;
        __syncthreads();   // the previous tile's readers and copiers are done
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int chunk = t + 256 * j;
            *reinterpret_cast<uint4 *>(tile + (chunk >> 4) * kQTPitch + (chunk & 15) * 16) = v[j];
        }
        __syncthreads();
        if (i + gridDim.x < n_tiles) {
            cur = locate(i + gridDim.x);
            load(cur);
        }
        // column c, blocks 2h and 2h + 1 (rows 64h .. 64h + 63)
        const int c = t & (kQT - 1);
        const int h = t >> 7;
        uint32_t codes = 0;
#pragma unroll 1
        for (int bb = 0; bb < 2; ++bb) {
            const int b = 2 * h + bb;
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                f[j] = __uint_as_float(
                    (uint32_t)*reinterpret_cast<const uint16_t *>(tile + (b * 32 + j) * kQTPitch +
                                                                  c * 2)
                    << 16);
            uint32_t w[8];
            codes |= mx_quantize_block(f, w) << (8 * bb);
            store_block(cqt + c * kQCPitch + b * 32, w);
        }
        // this tile's blocks 4 rt .. 4 rt + 3 of the group: bytes 4 (rt % 4) ..
        // of 16-byte slot sofs[g] / 16 + rt / 4
        const size_t slot = (size_t)(s_slot0[tl.g] + tl.rt / 4);
        *reinterpret_cast<uint16_t *>(sft + (slot * C + tl.c0 + c) * 16 + 4 * (tl.rt & 3) + 2 * h) =
            (uint16_t)codes;
        __syncthreads();
        // the code tile out: one contiguous 16 KB chunk (128 columns x 128 k)
        uint8_t *dst = qt + ((size_t)(s_tile0[tl.g] + tl.rt) * C + tl.c0) * kQT;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int chunk = t + 256 * j;
            const int row = chunk >> 3, c16 = (chunk & 7) * 16;
            *reinterpret_cast<uint4 *>(dst + (size_t)row * kQT + c16) =
                *reinterpret_cast<const uint4 *>(cqt + row * kQCPitch + c16);
        }
    }
}

}  // namespace

moe_status launch_mx_kpad_plan(const int32_t *offsets, int G, int32_t *kofs, int32_t *sofs,
                               cudaStream_t st) {
    if (G < 1) return MOE_ERR_INVALID_ARG;
    mx_kpad_plan_kernel<<<1, 32, 0, st>>>(offsets, G, kofs, sofs);
    return cuda_status(cudaGetLastError());
}

moe_status launch_mx_quantize_rows_t(const uint16_t *src, const int32_t *row_idx,
                                     const int32_t *offsets, const int32_t *kofs,
                                     const int32_t *sofs, int G, int max_tiles, int C,
                                     uint8_t *qt, uint8_t *sft, cudaStream_t st) {
    if (C % kQT != 0) return MOE_ERR_UNSUPPORTED;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    // the bf16 tile, one code tile and the groups' tables: three CTAs per SM
    const int smem = kQT * kQTPitch + kQT * kQCPitch + 3 * 4 * (G + 1);
    if (G > 1025) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(mx_quantize_rows_t_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kQT * kQTPitch + kQT * kQCPitch + 3 * 4 * 1026) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        attr_set[dev] = true;
    }
    const long long n = (long long)max_tiles * (C / kQT);
    if (n <= 0) return MOE_OK;
    const long long cap = (long long)num_sms() * 3;
    const int blocks = (int)(n < cap ? n : cap);
    mx_quantize_rows_t_kernel<<<blocks, 256, smem, st>>>(src, row_idx, offsets, kofs, sofs, G, C,
                                                         qt, sft);
    return cuda_status(cudaGetLastError());
}

moe_status launch_mx_quantize_both(const uint16_t *src, int G, int R, int C, uint8_t *q,
                                   uint8_t *sf, uint8_t *qt, uint8_t *sft, cudaStream_t st) {
    if (R % kQT != 0 || C % kQT != 0) return MOE_ERR_UNSUPPORTED;
    const long long n_tiles = (long long)G * (R / kQT) * (C / kQT);
    if (n_tiles == 0) return MOE_OK;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(mx_quantize_both_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        attr_set[dev] = true;
    }
    const long long cap = (long long)num_sms() * 3;
    const int blocks = (int)(n_tiles < cap ? n_tiles : cap);
    mx_quantize_both_kernel<<<blocks, 256, kQSmem, st>>>(src, G, R, C, mx_sf_pitch(C),
                                                         mx_sf_pitch(R), q, sf, qt, sft);
    return cuda_status(cudaGetLastError());
}

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

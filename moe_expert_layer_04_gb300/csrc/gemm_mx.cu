// gemm_mx.cu -- MXFP8 expert GEMMs: E4M3 operands with E8M0 scales per block
// of 32 along the contraction (OCP MX v1.0), on the bf16 tensor-core path.
//
//   MX GEMM 1   [g|u] = x~ W13~[g]^T,  h~ = MX(silu(min(g,c)) clamp(u,-c,c))
//   MX GEMM 2   y = w * (h~ W2~[g]^T)                               (bf16)
// ("DeepSeek-V4昇腾训练支持：基于 CANN 平台的TorchTitan-NPU + AutoFuse
// 极简训练优化实践", 性能结果与未来展望: FP8 training on MxFP8 compute; the
// expert matmuls themselves: "HyperParallel加速DeepSeek-V4.1多模态1M长序列
// 训练" §2.3 MegaMoE.)
//
// An E4M3 value times a power-of-two scale is an exact bf16 value, and the
// products of bf16 values are exact in the fp32 accumulator, so expanding
// both MX operands to bf16 in shared memory and running the bf16
// tcgen05.mma gives the sums of a block-scaled MXFP8 MMA up to the order of
// the fp32 additions.  The operands cross HBM at one byte per element plus
// one scale byte per 32, half the bytes of bf16; what bounds these GEMMs is
// the expansion itself (its instructions and its shared-memory traffic: per
// k-step 24 KB of codes read back and 48 KB of bf16 written, beside the
// tensor cores' 48 KB of operand reads).
//
// One CTA per SM, 18 warps:
//   warp 0      TMA producer: code tiles (A 128 x 64, B 256 x 64 bytes, 64-byte
//               swizzle) into a 4-stage ring; every 8 k-steps the scale codes
//               of the tile's rows for those 8 steps (16 bytes a row) into a
//               2-slot ring.
//   warp 1      TMEM owner and MMA issuer (bf16, M = 128, N = 256, K = 16;
//               two accumulators).
//   warps 2-5   epilogue, thread = row: GEMM 1 the clamped SwiGLU and h
//               quantised to MXFP8 per 32 columns (hardware conversion);
//               GEMM 2 the routing-weight scale to bf16.
//   warps 6-17  converters, three per scheduler: thread c expands row c of a
//               code stage (rows 0-127 A, 128-383 B) into a 128-byte-swizzled
//               bf16 stage (2 stages), then releases both.  Fewer warps leave
//               the schedulers idle on the conversion's dependency chains.
// Every wait is bounded; on a timeout the CTA records MOE_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and exits.
#include <cstring>

#include "gemm_launch.cuh"
#include "mx_common.cuh"

namespace moe {
namespace {

enum MxMode : int { MX_FFN1 = 0, MX_FFN2 = 1 };

struct MxParams {
    CUtensorMap tmA;   // A codes [rows, K] u8, boxes 64 x 128, 64-byte swizzle
    CUtensorMap tmB;   // B codes [G * b_rows_per_group, K] u8, same boxes
    CUtensorMap tmSA;  // A scale codes [rows, pitch] u8, boxes 16 x 128
    CUtensorMap tmSB;  // B scale codes [G * b_rows_per_group, pitch] u8
    const int32_t *offsets;
    int G;
    int n_tiles;           // column tiles per row tile
    int k_blocks;          // K / 64
    int b_rows_per_group;  // 2I (GEMM 1) or d (GEMM 2)
    int I;
    int N;                 // GEMM 2: output columns (d)
    float clamp;
    uint8_t *hq;           // GEMM 1: h codes [rows, I]
    uint8_t *hsf;          // GEMM 1: h scale codes [rows, h_pitch]
    int h_pitch;
    uint16_t *y;           // GEMM 2: [rows, d] bf16
    const float *row_w;    // GEMM 2: weight of rows < w_rows (others 1)
    int w_rows;
    int *status;
    long long wait_limit;
};

constexpr int kMxRaw = 4;           // code stages
constexpr int kMxBf = 2;            // bf16 operand stages
constexpr int kMxSfSlots = 2;       // scale slots (8 k-steps each)
constexpr int kMxEpiWarps = 4;
constexpr int kMxConvWarps = 12;    // one A or B row per thread
constexpr int kMxThreads = 64 + 32 * (kMxEpiWarps + kMxConvWarps);
constexpr int kMxRawA = 128 * 64;
constexpr int kMxRawStage = kMxRawA + 256 * 64;
constexpr int kMxBfA = 128 * 128;
constexpr int kMxBfStage = kMxBfA + 256 * 128;
constexpr int kMxSfA = 128 * 16;
constexpr int kMxSfSlot = kMxSfA + 256 * 16;
constexpr int kMxBarBytes = 256;
constexpr int kMxFixedSmem = kMxBf * kMxBfStage + kMxRaw * kMxRawStage + kMxSfSlots * kMxSfSlot;
static_assert((2 * kMxRaw + 2 * kMxBf + 2 * kMxSfSlots + 5) * 8 + 8 <= kMxBarBytes,
              "barrier block");

inline size_t mx_smem_bytes(int G) {
    return 1024 + (size_t)kMxFixedSmem + kMxBarBytes + 8 * (size_t)(G + 2);
}

__device__ __forceinline__ TileInfo mx_tile(const MxParams &p, int t, const int *mt_start,
                                            const int *offs) {
    TileInfo ti{};
    ti.nt = t % p.n_tiles;
    const int q = t / p.n_tiles;
    int lo = 0, hi = p.G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mt_start[mid] <= q) lo = mid; else hi = mid - 1;
    }
    ti.g = lo;
    ti.row0 = offs[lo] + (q - mt_start[lo]) * 128;
    ti.rows_valid = min(128, offs[lo + 1] - ti.row0);
    ti.kb = p.k_blocks;
    ti.rt = q;
    return ti;
}

// Row r of a code tile (64 bytes, 64-byte swizzle) -> row r of a bf16 tile
// (128 bytes, 128-byte swizzle; inside each group of four contraction
// elements the order 0, 2, 1, 3, the same for A and B rows); elements 0-31
// scaled by 2^(sf[0] - 127), 32-63 by 2^(sf[1] - 127).
template <bool TWO>
__device__ __forceinline__ void mx_expand_row_t(const uint8_t *codes, const MxBf16Factors &f0,
                                                const MxBf16Factors &f1, uint8_t *dst, int r) {
    const uint32_t sw_in = (uint32_t)(r >> 1) & 3u;
    const uint32_t sw = (uint32_t)r & 7u;
    const uint8_t *src = codes + r * 64;
    const uint32_t out = smem_u32(dst + r * 128);
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(src + ((c ^ sw_in) << 4));
        const MxBf16Factors &f = c < 2 ? f0 : f1;
        uint32_t o[8];
        e4m3x4_to_bf16x2x2<TWO>(v.x, f, o[0], o[1]);
        e4m3x4_to_bf16x2x2<TWO>(v.y, f, o[2], o[3]);
        e4m3x4_to_bf16x2x2<TWO>(v.z, f, o[4], o[5]);
        e4m3x4_to_bf16x2x2<TWO>(v.w, f, o[6], o[7]);
        st_shared_v4(out + (((2 * c) ^ sw) << 4), o[0], o[1], o[2], o[3]);
        st_shared_v4(out + (((2 * c + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
    }
}

// One decision per row and k-step: the second multiply only where a block's
// scale exceeds 2^7 (rare), so the common path carries no per-word test.
__device__ __forceinline__ void mx_expand_row(const uint8_t *codes, const uint8_t *sf,
                                              uint8_t *dst, int r) {
    const MxBf16Factors f0 = mx_bf16_factors(sf[0]);
    const MxBf16Factors f1 = mx_bf16_factors(sf[1]);
    if (f0.two || f1.two) mx_expand_row_t<true>(codes, f0, f1, dst, r);
    else mx_expand_row_t<false>(codes, f0, f1, dst, r);
}

template <int MODE>
__global__ void __launch_bounds__(kMxThreads, 1) moe_mx_gemm_kernel(const __grid_constant__ MxParams p) {
    constexpr uint32_t IDESC = idesc_bf16_f32(128, 256, false, false);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sBf = smem;
    uint8_t *sRaw = smem + kMxBf * kMxBfStage;
    uint8_t *sSf = sRaw + kMxRaw * kMxRawStage;
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smem + kMxFixedSmem);
    uint64_t *rempty = rfull + kMxRaw;
    uint64_t *bfull = rempty + kMxRaw;
    uint64_t *bempty = bfull + kMxBf;
    uint64_t *sfull = bempty + kMxBf;
    uint64_t *sempty = sfull + kMxSfSlots;
    uint64_t *tfull = sempty + kMxSfSlots;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_s = reinterpret_cast<volatile int *>(tmem_base_s + 1);
    int *offs = reinterpret_cast<int *>(smem + kMxFixedSmem + kMxBarBytes);
    int *mt_start = offs + (p.G + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxRaw; ++s) {
            mbar_init(&rfull[s], 1);
            mbar_init(&rempty[s], kMxConvWarps);
        }
        for (int s = 0; s < kMxBf; ++s) {
            mbar_init(&bfull[s], kMxConvWarps);
            mbar_init(&bempty[s], 1);
        }
        for (int s = 0; s < kMxSfSlots; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], kMxConvWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 32 * kMxEpiWarps);
        }
        mbar_init(done, 1);
        *abort_s = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(&p.tmB);
        tma_prefetch_desc(&p.tmSA);
        tma_prefetch_desc(&p.tmSB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_s, 512);
        tmem_relinquish();
    }
    if (warp == 2) {
        // group offsets and the exclusive prefix of their 128-row tiles
        int carry = 0;
        for (int base = 0; base <= p.G; base += 32) {
            const int g = base + lane;
            int o = 0;
            if (g <= p.G) {
                o = p.offsets[g];
                offs[g] = o;
            }
            int mt = 0;
            if (g < p.G) {
                const int cnt = p.offsets[g + 1] - o;
                mt = cnt > 0 ? (cnt + 127) >> 7 : 0;
            }
            int incl = mt;
#pragma unroll
            for (int sft = 1; sft < 32; sft <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, sft);
                if (lane >= sft) incl += v;
            }
            if (g <= p.G) mt_start[g] = carry + incl - mt;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_base_s;
    const WaitCtl wc{abort_s, p.status, p.wait_limit};
    const int total_tiles = mt_start[p.G] * p.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_r[kMxRaw], last_s[kMxSfSlots];
#pragma unroll
            for (int i = 0; i < kMxRaw; ++i) last_r[i] = -1;
#pragma unroll
            for (int i = 0; i < kMxSfSlots; ++i) last_s[i] = -1;
            uint32_t s = 0, ph = 0, js = 0, phs = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const TileInfo ti = mx_tile(p, t, mt_start, offs);
                // B rows of the tile: GEMM 1 the gate rows and the up rows of
                // its 128 h columns, GEMM 2 256 consecutive output rows
                const int brow = ti.g * p.b_rows_per_group + ti.nt * (MODE == MX_FFN1 ? 128 : 256);
                const int brow2 = MODE == MX_FFN1 ? brow + p.I : brow + 128;
                for (int kb = 0; kb < ti.kb; ++kb) {
                    if ((kb & 7) == 0) {
                        if (!mbar_wait(&sempty[js], phs ^ 1u, wc)) { ok = false; break; }
                        mbar_arrive_expect_tx(&sfull[js], kMxSfSlot);
                        uint8_t *d = sSf + js * kMxSfSlot;
                        const int x = (kb >> 3) * 16;
                        tma_load_2d(d, &p.tmSA, &sfull[js], x, ti.row0);
                        tma_load_2d(d + kMxSfA, &p.tmSB, &sfull[js], x, brow);
                        tma_load_2d(d + kMxSfA + 128 * 16, &p.tmSB, &sfull[js], x, brow2);
                        last_s[js] = (int)phs;
                        if (++js == kMxSfSlots) { js = 0; phs ^= 1u; }
                    }
                    if (!mbar_wait(&rempty[s], ph ^ 1u, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&rfull[s], kMxRawStage);
                    uint8_t *a = sRaw + s * kMxRawStage;
                    tma_load_2d(a, &p.tmA, &rfull[s], kb * 64, ti.row0);
                    tma_load_2d(a + kMxRawA, &p.tmB, &rfull[s], kb * 64, brow);
                    tma_load_2d(a + kMxRawA + 128 * 64, &p.tmB, &rfull[s], kb * 64, brow2);
                    last_r[s] = (int)ph;
                    if (++s == kMxRaw) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // drain the copies still in flight before the CTA exits
                for (int i = 0; i < kMxRaw; ++i)
                    if (last_r[i] >= 0) mbar_wait_teardown(&rfull[i], (uint32_t)last_r[i], p.wait_limit);
                for (int i = 0; i < kMxSfSlots; ++i)
                    if (last_s[i] >= 0) mbar_wait_teardown(&sfull[i], (uint32_t)last_s[i], p.wait_limit);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        uint32_t sb = 0, phb = 0;
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, ++it) {
            const TileInfo ti = mx_tile(p, t, mt_start, offs);
            const uint32_t acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(&tempty[acc], aph ^ 1u, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * 256;
            for (int kb = 0; kb < ti.kb; ++kb) {
                if (!mbar_wait(&bfull[sb], phb, wc)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_addr = smem_u32(sBf + sb * kMxBfStage);
                    const uint32_t b_addr = a_addr + kMxBfA;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(d_tmem, sdesc_sw128(a_addr + kk * 32, 16, 1024),
                                  sdesc_sw128(b_addr + kk * 32, 16, 1024), IDESC,
                                  (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(&bempty[sb]);
                }
                __syncwarp();
                if (++sb == kMxBf) { sb = 0; phb ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&tfull[acc]);
            __syncwarp();
        }
        if (!ok) {
            // every MMA this thread issued must finish before TMEM is freed
            if (lane == 0) umma_commit(done);
            __syncwarp();
            mbar_wait_teardown(done, 0, p.wait_limit);
        }
    } else if (warp >= 2 + kMxEpiWarps) {
        // ------------------------------------------------ converters
        // rows 0..127: A, 128..383: B; warps hold one kind of row each
        const int ct = (warp - 2 - kMxEpiWarps) * 32 + lane;   // 0..383
        const bool is_a = ct < 128;
        const int r = is_a ? ct : ct - 128;
        uint32_t s = 0, ph = 0, sb = 0, phb = 0, js = 0, phs = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
            const TileInfo ti = mx_tile(p, t, mt_start, offs);
            for (int kb = 0; kb < ti.kb; ++kb) {
                if ((kb & 7) == 0 && !mbar_wait(&sfull[js], phs, wc)) { ok = false; break; }
                if (!mbar_wait(&rfull[s], ph, wc)) { ok = false; break; }
                if (!mbar_wait(&bempty[sb], phb ^ 1u, wc)) { ok = false; break; }
                const uint8_t *raw = sRaw + s * kMxRawStage;
                const uint8_t *sf = sSf + js * kMxSfSlot + (kb & 7) * 2;
                uint8_t *bf = sBf + sb * kMxBfStage;
                // A rows past the group's end feed only accumulator rows that are
                // never stored (MMA rows are independent), so they are not expanded
                if (!is_a) mx_expand_row(raw + kMxRawA, sf + kMxSfA + r * 16, bf + kMxBfA, r);
                else if (r < ti.rows_valid) mx_expand_row(raw, sf + r * 16, bf, r);
                // the tensor cores read the stage through the async proxy
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bfull[sb]);
                    mbar_arrive(&rempty[s]);
                }
                if (++s == kMxRaw) { s = 0; ph ^= 1u; }
                if (++sb == kMxBf) { sb = 0; phb ^= 1u; }
                if ((kb & 7) == 7 || kb == ti.kb - 1) {
                    if (lane == 0) mbar_arrive(&sempty[js]);
                    if (++js == kMxSfSlots) { js = 0; phs ^= 1u; }
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int q = warp & 3;   // TMEM lane quadrant this warp may read
        const int r_local = q * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
            const TileInfo ti = mx_tile(p, t, mt_start, offs);
            const uint32_t acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(&tfull[acc], aph, wc)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256;
            const bool valid = r_local < ti.rows_valid;
            const int row = ti.row0 + r_local;
            if constexpr (MODE == MX_FFN1) {
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t rg[32], ru[32];
                    tmem_ld32(tb + c, rg);
                    tmem_ld32(tb + 128 + c, ru);
                    tmem_wait_ld();
                    if (valid) {
                        float hv[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            hv[j] = swiglu_clamped(__uint_as_float(rg[j]), __uint_as_float(ru[j]),
                                                   p.clamp);
                        uint32_t w[8];
                        const uint32_t code = mx_quantize_block_hw(hv, w);
                        const int col = ti.nt * 128 + c;
                        uint8_t *dst = p.hq + (size_t)row * p.I + col;
                        st_global_v4(dst, w[0], w[1], w[2], w[3]);
                        st_global_v4(dst + 16, w[4], w[5], w[6], w[7]);
                        p.hsf[(size_t)row * p.h_pitch + col / 32] = (uint8_t)code;
                    }
                }
            } else {
                float w = 1.0f;
                if (valid && p.row_w && row < p.w_rows) w = p.row_w[row];
                epi_bf16_scaled<256>(p.y, p.N, ti, tb, valid, row, w);
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <int MODE>
moe_status launch_mx(MxParams &p, int max_tiles, cudaStream_t st) {
    auto kern = moe_mx_gemm_kernel<MODE>;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mx_smem_bytes(kMaxGroups)) != cudaSuccess)
            return MOE_ERR_CUDA;
        attr_set[dev] = true;
    }
    if (max_tiles <= 0) return MOE_OK;
    p.status = device_status_ptr();
    if (!p.status) return MOE_ERR_CUDA;
    if (p.wait_limit <= 0) p.wait_limit = kWaitLimitCycles;
    const int grid = max_tiles < num_sms() ? max_tiles : num_sms();
    kern<<<grid, kMxThreads, mx_smem_bytes(p.G), st>>>(p);
    return cuda_status(cudaGetLastError());
}

}  // namespace

moe_status launch_mx_ffn1(const uint8_t *xq, const uint8_t *xsf, const int32_t *offsets, int G,
                          int max_rows, const uint8_t *W13q, const uint8_t *W13sf, int d, int I,
                          float clamp, uint8_t *hq, uint8_t *hsf, cudaStream_t st) {
    if (d % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    MxParams p;
    std::memset(&p, 0, sizeof p);
    const int sfd = mx_sf_pitch(d);
    const uint64_t brows = (uint64_t)G * 2 * I;
    if (!encode_tmap_u8_2d(&p.tmA, xq, d, max_rows, d, 64, 128, 64) ||
        !encode_tmap_u8_2d(&p.tmB, W13q, d, brows, d, 64, 128, 64) ||
        !encode_tmap_u8_2d(&p.tmSA, xsf, sfd, max_rows, sfd, 16, 128, 0) ||
        !encode_tmap_u8_2d(&p.tmSB, W13sf, sfd, brows, sfd, 16, 128, 0))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = I / 128;
    p.k_blocks = d / 64;
    p.b_rows_per_group = 2 * I;
    p.I = I;
    p.clamp = clamp;
    p.hq = hq;
    p.hsf = hsf;
    p.h_pitch = mx_sf_pitch(I);
    return launch_mx<MX_FFN1>(p, row_tile_bound(max_rows, G) * p.n_tiles, st);
}

moe_status launch_mx_ffn2(const uint8_t *hq, const uint8_t *hsf, const int32_t *offsets, int G,
                          int max_rows, const uint8_t *W2q, const uint8_t *W2sf,
                          const float *row_w, int S, int d, int I, uint16_t *y, cudaStream_t st) {
    if (d % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    MxParams p;
    std::memset(&p, 0, sizeof p);
    const int sfi = mx_sf_pitch(I);
    const uint64_t brows = (uint64_t)G * d;
    if (!encode_tmap_u8_2d(&p.tmA, hq, I, max_rows, I, 64, 128, 64) ||
        !encode_tmap_u8_2d(&p.tmB, W2q, I, brows, I, 64, 128, 64) ||
        !encode_tmap_u8_2d(&p.tmSA, hsf, sfi, max_rows, sfi, 16, 128, 0) ||
        !encode_tmap_u8_2d(&p.tmSB, W2sf, sfi, brows, sfi, 16, 128, 0))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = d / 256;
    p.k_blocks = I / 64;
    p.b_rows_per_group = d;
    p.I = I;
    p.N = d;
    p.y = y;
    p.row_w = row_w;
    p.w_rows = S;
    return launch_mx<MX_FFN2>(p, row_tile_bound(max_rows, G) * p.n_tiles, st);
}

}  // namespace moe

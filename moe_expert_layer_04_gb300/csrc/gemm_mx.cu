// gemm_mx.cu -- MXFP8 expert GEMMs: E4M3 operands with E8M0 scales per block
// of 32 along the contraction (OCP MX v1.0), on the block-scaled tensor-core
// MMA (tcgen05.mma kind::mxf8f6f4).
//
//   MX GEMM 1   [g|u] = x~ W13~[g]^T,  h~ = MX(silu(min(g,c)) clamp(u,-c,c))
//               (and the fp32 g|u for the backward, when it is saved)
//   MX GEMM 2   y = w * (h~ W2~[g]^T)                               (bf16)
//   MX dgrad 2  dA = dY~ (W2^T)~[g]^T, with W2 quantised along d; epilogue:
//               the partial <h~, dA> per tile, dH = w dA through the clamped
//               SwiGLU's derivative -> dG|dU (bf16, and MX along 2I), w h~
//               (bf16)
//   MX dgrad 1  dX = dGU~ (W13^T)~[g]^T, with W13 quantised along 2I: GEMM 2
//               with K = 2I and no row weight
//   MX wgrad    dW[g] = A~^T B~ over group g's rows, both operands quantised
//               along the rows (blocks of 32 from the group's first row,
//               padded to 128) and stored transposed, K-chunk-major (each
//               stage one contiguous 16 KB box); fp32 out through TMA stores
// ("DeepSeek-V4昇腾训练支持：基于 CANN 平台的TorchTitan-NPU + AutoFuse 极简训练优化
// 实践", 性能结果与未来展望: FP8 training on MxFP8 compute; the expert matmuls
// themselves: "HyperParallel加速DeepSeek-V4.1多模态1M长序列训练" §2.3 MegaMoE.)
//
// The tensor cores read the E4M3 codes straight from shared memory and apply
// each block's scale from tensor memory, so every product is exact and the
// sums are fp32: the results are those of the MX definition up to the order
// of the fp32 additions.  The operands cross HBM at one byte an element plus
// one scale byte per 32.
//
// Tiles are 128 rows x BN columns (GEMM 1: BN/2 gate and the matching BN/2
// up columns, i.e. BN/2 h columns; GEMM 2: BN output columns), 128
// contraction elements per stage.  BN = 128: two fp32 accumulators (one
// tile's epilogue overlaps the next tile's MMAs), for few rows per expert,
// where the weights stream from HBM.  BN = 256: one accumulator (512 tensor
// memory columns would leave none for the scales), half the operand bytes per
// MMA from L2, for many rows per expert, where the MMAs set the pace.  Per
// stage tensor memory also holds four columns of A scales and BN/32 of B
// scales.  Each of the four lane
// quadrants computes its 32 rows of D against every column, so it reads the
// scales of all of B, and of A, from its own lanes: in every quadrant q, lane
// 32q + j at column (first + c) holds the word of row 32c + j; the
// instruction descriptor picks its byte -- byte j for the j-th block of 32 of
// the stage.
//
// One CTA per SM, 10 warps (14 with two epilogue warps per lane quadrant:
// the 256-wide tiles and dgrad 2):
//   warp 0      TMA producer: per stage the A and B code tiles (128-byte rows,
//               128-byte swizzle), per four stages the 16-byte scale rows of
//               A and B that hold their scale codes.
//   warp 1      TMEM owner and MMA issuer (block-scaled MMA, M = 128,
//               N = BN, K = 32, four per stage).
//   warps 2-    epilogue, thread = row: GEMM 1 the clamped SwiGLU and h
//               quantised to MXFP8 per 32 columns (hardware conversion);
//               GEMM 2 the routing-weight scale to bf16; dgrad 2 the SwiGLU
//               backward and its four outputs.
//   last 4      scale writers, one per TMEM lane quadrant, thread = row: per
//               stage the four A scale codes and the B scale codes of its
//               rows into tensor memory (tcgen05.st), then the stage is
//               released to the MMA issuer.  (Loading a slot's 16-byte rows
//               once into registers and releasing the slot early measured
//               slower for the forward GEMMs and dgrad 1.)
// Every wait is bounded; on a timeout the CTA records MOE_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and exits.
#include <cstring>

#include <cuda_fp16.h>

#include "gemm_launch.cuh"
#include "mx_common.cuh"

namespace moe {
namespace {

enum MxMode : int { MX_FFN1 = 0, MX_FFN2 = 1, MX_DGRAD2 = 2, MX_WGRAD = 3 };

struct MxParams {
    CUtensorMap tmA;   // A codes [rows, K] u8, boxes 128 x 128, 128-byte swizzle
    CUtensorMap tmO;   // dgrad 2: dG|dU [rows, 2I] bf16, boxes 32 x 32, 64-byte swizzle
    CUtensorMap tmO2;  // dgrad 2: w h~ [rows, I] bf16, boxes 32 x 32, 64-byte swizzle
    CUtensorMap tmOQ;  // dgrad 2: dG|dU codes [rows, 2I] u8, boxes 32 x 32
                       // weight gradients: fp32 output [G * M, N], boxes 32 x 32
    CUtensorMap tmB;   // B codes [G * b_rows_per_group, K] u8, boxes 128 x 64 (GEMM 1) / 128 x 128
    CUtensorMap tmSA;  // A scale codes [rows, pitch] u8, boxes 16 x 128
    CUtensorMap tmSB;  // B scale codes, boxes 16 x 64 (GEMM 1) / 16 x 128
    const int32_t *offsets;
    int G;
    int n_tiles;           // column tiles per row tile
    int k_blocks;          // K / 128
    int b_rows_per_group;  // 2I (GEMM 1) or d (GEMM 2)
    int I;
    int N;                 // GEMM 2: output columns (d)
    float clamp;
    uint8_t *hq;           // GEMM 1: h codes [rows, I]
    uint8_t *hsf;          // GEMM 1: h scale codes [rows, h_pitch]
    int h_pitch;
    float *gu_out;         // GEMM 1: fp32 g|u (gu_offset layout) or null
    uint16_t *y;           // GEMM 2: [rows, d] bf16
    const float *row_w;    // GEMM 2, dgrad 2: weight of rows < w_rows (others 1)
    int w_rows;
    const float *gu_in;    // dgrad 2: the forward's fp32 g|u (gu_offset layout)
    const uint8_t *hq_in;  // dgrad 2: the forward's h~ codes [rows, I] ...
    const uint8_t *hsf_in; //          ... and scale codes [rows, h_pitch]
    uint16_t *dgu;         // dgrad 2: dG|dU [rows, 2I] bf16
    uint8_t *dguq;         //          dG|dU MX along 2I: codes [rows, 2I] ...
    uint8_t *dgusf;        //          ... and scale codes [rows, dgu_pitch]
    int dgu_pitch;
    uint16_t *hw;          // dgrad 2: w h~ [rows, I] bf16
    float *dw_part;        // dgrad 2: [rows, n_tiles * NEPI / 4] partials of <h~, dA>
    int M;                 // weight gradients: output rows per group (A rows)
    const int32_t *sofs;   // weight gradients: [G+1] first scale byte of each group
                           // (offsets holds the first code column, kofs)
    // weight gradients and dgrad 2: tiles handed out at run time (as in the
    // bf16 grouped GEMM) from this counter, zero before the launch; the
    // weight gradients take the groups in korder (longest contraction first)
    int *tile_counter;
    const int32_t *korder;
    int *status;
    long long wait_limit;
};

constexpr int kMxSfRow = 16;          // bytes of a scale row in a slot (4 stages' codes)
constexpr int kMxCodeA = 128 * 128;   // A codes of a stage
constexpr int kMxSfA = 128 * kMxSfRow;
constexpr int kMxSfWarps = 4;
constexpr int kMxSfSlots = 2;         // scale slots, 4 stages each
constexpr int kMxBarBytes = 512;
// weight gradients: operand stages, and fp32 staging blocks per epilogue warp
// (two let a block be staged while the previous one's TMA store reads)
constexpr int kMxWgradStages = 5;
constexpr int kMxWgradStageBufs = 2;
constexpr uint32_t kMxTmemCols = 512;

template <int MODE, int BN>
struct MxShape {
    static constexpr int CODE_B = BN * 128;
    static constexpr int STAGE = kMxCodeA + CODE_B;              // codes of a stage
    static constexpr int SF_SLOT = kMxSfA + BN * kMxSfRow;        // scales of 4 stages
    // the weight gradients' tiles have short contractions (a group's rows):
    // more stages keep more copies in flight
    static constexpr int STAGES = MODE == MX_WGRAD ? kMxWgradStages : 4;
    static constexpr int NACC = BN == 256 ? 1 : 2;                // accumulators
    // epilogue warps: two per lane quadrant for the wide tiles and for the
    // heavy epilogue of dgrad 2
    static constexpr int NEPI = (BN == 256 || MODE == MX_DGRAD2) ? 8 : 4;
    static constexpr int THREADS = 64 + 32 * (NEPI + kMxSfWarps);
    static constexpr uint32_t SF_COL0 = NACC * BN;                // scale columns after them
    static constexpr uint32_t SF_COLS = 4 + BN / 32;              // per stage: A, then B
    // dgrad 2: per epilogue warp one staging block for each of its five
    // outputs of 32 rows x 32 columns (dg, du, w h~ in bf16; dg, du codes)
    static constexpr int EPI_WARP = 3 * 2048 + 2 * 1024;
    static constexpr int EPI = MODE == MX_DGRAD2 ? NEPI * EPI_WARP
                               : MODE == MX_WGRAD ? NEPI * 4096 * kMxWgradStageBufs
                                                  : 0;
    static constexpr int FIXED = STAGES * STAGE + kMxSfSlots * SF_SLOT + EPI;
    static_assert(SF_COL0 + SF_COLS * STAGES <= kMxTmemCols, "tensor memory columns");
    static_assert((4 * STAGES + 2 * kMxSfSlots + 5 + 2 * kSchedSlots) * 8 + 8 + 4 * kSchedSlots <=
                      kMxBarBytes,
                  "barrier block");
};

template <int MODE, int BN>
inline size_t mx_smem_bytes(int G) {
    return 1024 + (size_t)MxShape<MODE, BN>::FIXED + kMxBarBytes + 8 * (size_t)(G + 2);
}

// Values of four E4M3 codes (one 32-bit word, element i in byte i), exact:
// the hardware conversion to f16 pairs (every E4M3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_values(uint32_t w, float (&v)[4]) {
    uint32_t lo, hi;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((uint16_t)(w & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((uint16_t)(w >> 16)));
    const __half2 l = *reinterpret_cast<const __half2 *>(&lo);
    const __half2 h = *reinterpret_cast<const __half2 *>(&hi);
    v[0] = __low2float(l);
    v[1] = __high2float(l);
    v[2] = __low2float(h);
    v[3] = __high2float(h);
}

template <int MODE>
__device__ __forceinline__ TileInfo mx_tile(const MxParams &p, int t, const int *mt_start,
                                            const int *offs) {
    TileInfo ti{};
    ti.nt = t % p.n_tiles;
    const int q = t / p.n_tiles;
    if constexpr (MODE == MX_WGRAD) {
        // (group, 128 output rows, BN output columns); the contraction is the
        // group's padded rows: code columns [offs[g], offs[g + 1]), scale
        // bytes from mt_start[g]
        const int mp = p.M / 128;
        const int qg = q / mp;   // the group's rank in the schedule
        ti.g = p.korder ? p.korder[qg] : qg;
        ti.m0 = (q - qg * mp) * 128;
        ti.krow0 = offs[ti.g];
        ti.krows = mt_start[ti.g];
        ti.kb = (offs[ti.g + 1] - offs[ti.g]) / 128;
        ti.row0 = ti.m0;
        ti.rows_valid = 128;
        return ti;
    }
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

template <int MODE, int BN>
__global__ void __launch_bounds__(MxShape<MODE, BN>::THREADS, 1)
    moe_mx_gemm_kernel(const __grid_constant__ MxParams p) {
    using SH = MxShape<MODE, BN>;
    constexpr int STAGES = SH::STAGES;
    constexpr int NACC = SH::NACC;
    constexpr int NEPI = SH::NEPI;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sCodes = smem;                                   // STAGES x (A | B codes)
    uint8_t *sSf = smem + STAGES * SH::STAGE;                 // kMxSfSlots x (A | B scales)
    uint8_t *sEpi = sSf + kMxSfSlots * SH::SF_SLOT;           // dgrad 2 staging (1 KB aligned)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SH::FIXED);
    uint64_t *empty = full + STAGES;      // the stage's MMAs are done (codes and scales free)
    uint64_t *sfready = empty + STAGES;   // the stage's scales are in tensor memory
    uint64_t *spare = sfready + STAGES;   // (unused; keeps the block layout simple)
    uint64_t *sffull = spare + STAGES;    // a scale slot landed
    uint64_t *sfempty = sffull + kMxSfSlots;   // the scale writers are done with a slot
    uint64_t *tfull = sfempty + kMxSfSlots;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    uint64_t *sfull = done + 1;              // ring of run-time tile indices
    uint64_t *sempty = sfull + kSchedSlots;
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(sempty + kSchedSlots);
    volatile int *abort_s = reinterpret_cast<volatile int *>(tmem_base_s + 1);
    volatile int *sched = abort_s + 1;
    int *offs = reinterpret_cast<int *>(smem + SH::FIXED + kMxBarBytes);
    int *mt_start = offs + (p.G + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sfready[s], kMxSfWarps);
            mbar_init(&spare[s], 1);
        }
        for (int j = 0; j < kMxSfSlots; ++j) {
            mbar_init(&sffull[j], 1);
            mbar_init(&sfempty[j], kMxSfWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 32 * NEPI);
        }
        mbar_init(done, 1);
        for (int j = 0; j < kSchedSlots; ++j) {
            mbar_init(&sfull[j], 1);
            // readers: the MMA issuer, the scale writers and the epilogue warps
            mbar_init(&sempty[j], 1 + kMxSfWarps + NEPI);
        }
        *abort_s = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(&p.tmB);
        tma_prefetch_desc(&p.tmSA);
        tma_prefetch_desc(&p.tmSB);
        if constexpr (MODE == MX_DGRAD2) {
            tma_prefetch_desc(&p.tmO);
            tma_prefetch_desc(&p.tmO2);
            tma_prefetch_desc(&p.tmOQ);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_s, kMxTmemCols);
        tmem_relinquish();
    }
    if (MODE == MX_WGRAD && warp == 2) {
        // the groups' code column and scale byte offsets
        for (int g = lane; g <= p.G; g += 32) {
            offs[g] = p.offsets[g];
            mt_start[g] = p.sofs[g];
        }
    } else if (warp == 2) {
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
    const int total_tiles =
        MODE == MX_WGRAD ? p.G * (p.M / 128) * p.n_tiles : mt_start[p.G] * p.n_tiles;

    // Run-time tile order (the weight gradients and dgrad 2, when the launcher
    // passes a counter): the producer takes each index from the counter and
    // passes it to the other roles through the ring, as in the bf16 grouped
    // GEMM, so the tiles in flight stay a window of about one per CTA and
    // share their operand rows in L2.  Otherwise a static round robin.
    const bool DYN = (MODE == MX_WGRAD || MODE == MX_DGRAD2) && p.tile_counter != nullptr;
    auto next_tile = [&](int i, bool writer, uint32_t mask) -> int {
        if (!DYN) return blockIdx.x + i * gridDim.x;
        const int j = i % kSchedSlots;
        const uint32_t sp = (uint32_t)(i / kSchedSlots) & 1u;
        if (writer) {
            if (!mbar_wait(&sempty[j], sp ^ 1u, wc)) return -1;
            int t = atomicAdd(p.tile_counter, 1);
            if (t > total_tiles) t = total_tiles;
            sched[j] = t;
            mbar_arrive(&sfull[j]);
            return t;
        }
        if (!mbar_wait(&sfull[j], sp, wc)) return -1;
        const int t = sched[j];
        __syncwarp(mask);
        // the arrival depends on the index read, so it cannot pass that read
        if (lane == 0 && t >= 0) mbar_arrive(&sempty[j]);
        return t;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_par[STAGES], last_sf[kMxSfSlots];
#pragma unroll
            for (int i = 0; i < STAGES; ++i) last_par[i] = -1;
#pragma unroll
            for (int i = 0; i < kMxSfSlots; ++i) last_sf[i] = -1;
            uint32_t s = 0, ph = 0, js = 0, phs = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int t = next_tile(i, true, 1u);
                if (t < 0) { ok = false; break; }
                if (t >= total_tiles) break;
                const TileInfo ti = mx_tile<MODE>(p, t, mt_start, offs);
                // B rows of the tile: GEMM 1 the gate rows and the up rows of its
                // BN/2 h columns, GEMM 2 BN consecutive output rows
                const int brow = ti.g * p.b_rows_per_group + ti.nt * (MODE == MX_FFN1 ? BN / 2 : BN);
                // weight gradients (K-chunk-major operands): the group's first
                // chunk of 128 codes and first 16-byte scale slot
                const int kc0 = MODE == MX_WGRAD ? ti.krow0 / 128 : 0;
                const int ks0 = MODE == MX_WGRAD ? ti.krows / kMxSfRow : 0;
                for (int kb = 0; kb < ti.kb; ++kb) {
                    if ((kb & 3) == 0) {
                        // the scale codes of this and the next three stages (16 bytes a row)
                        if (!mbar_wait(&sfempty[js], phs ^ 1u, wc)) { ok = false; break; }
                        mbar_arrive_expect_tx(&sffull[js], SH::SF_SLOT);
                        uint8_t *sa = sSf + js * SH::SF_SLOT;
                        uint8_t *sb = sa + kMxSfA;
                        const int x = (kb >> 2) * kMxSfRow;
                        if constexpr (MODE == MX_WGRAD) {
                            const int slot = ks0 + (kb >> 2);
                            tma_load_2d(sa, &p.tmSA, &sffull[js], 0, slot * p.M + ti.m0);
                            tma_load_2d(sb, &p.tmSB, &sffull[js], 0, slot * p.N + brow);
                        } else {
                            tma_load_2d(sa, &p.tmSA, &sffull[js], x, ti.row0);
                        }
                        if constexpr (MODE == MX_WGRAD) {
                        } else if constexpr (MODE == MX_FFN1) {
                            tma_load_2d(sb, &p.tmSB, &sffull[js], x, brow);
                            tma_load_2d(sb + (BN / 2) * kMxSfRow, &p.tmSB, &sffull[js], x,
                                        brow + p.I);
                        } else {
                            tma_load_2d(sb, &p.tmSB, &sffull[js], x, brow);
                        }
                        last_sf[js] = (int)phs;
                        if (++js == kMxSfSlots) { js = 0; phs ^= 1u; }
                    }
                    if (!mbar_wait(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], SH::STAGE);
                    uint8_t *a = sCodes + s * SH::STAGE;
                    uint8_t *b = a + kMxCodeA;
                    if constexpr (MODE == MX_WGRAD) {
                        const int kc = kc0 + kb;
                        tma_load_2d(a, &p.tmA, &full[s], 0, kc * p.M + ti.m0);
                        tma_load_2d(b, &p.tmB, &full[s], 0, kc * p.N + brow);
                    } else if constexpr (MODE == MX_FFN1) {
                        tma_load_2d(a, &p.tmA, &full[s], kb * 128, ti.row0);
                        tma_load_2d(b, &p.tmB, &full[s], kb * 128, brow);
                        tma_load_2d(b + (BN / 2) * 128, &p.tmB, &full[s], kb * 128, brow + p.I);
                    } else {
                        tma_load_2d(a, &p.tmA, &full[s], kb * 128, ti.row0);
                        tma_load_2d(b, &p.tmB, &full[s], kb * 128, brow);
                    }
                    last_par[s] = (int)ph;
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // drain the copies still in flight before the CTA exits
                for (int i = 0; i < STAGES; ++i)
                    if (last_par[i] >= 0)
                        mbar_wait_teardown(&full[i], (uint32_t)last_par[i], p.wait_limit);
                for (int i = 0; i < kMxSfSlots; ++i)
                    if (last_sf[i] >= 0)
                        mbar_wait_teardown(&sffull[i], (uint32_t)last_sf[i], p.wait_limit);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        uint32_t s = 0, ph = 0;
        int it = 0;
        bool ok = true;
        for (; ok; ++it) {
            const int t = next_tile(it, false, 0xffffffffu);
            if (t < 0) { ok = false; break; }
            if (t >= total_tiles) break;
            const TileInfo ti = mx_tile<MODE>(p, t, mt_start, offs);
            const uint32_t acc = NACC == 2 ? (it & 1) : 0;
            const uint32_t aph = NACC == 2 ? ((it >> 1) & 1) : (it & 1);
            if (!mbar_wait(&tempty[acc], aph ^ 1u, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < ti.kb; ++kb) {
                if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
                if (!mbar_wait(&sfready[s], ph, wc)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_addr = smem_u32(sCodes + s * SH::STAGE);
                    const uint32_t b_addr = a_addr + kMxCodeA;
                    const uint32_t sfa = tmem_base + SH::SF_COL0 + SH::SF_COLS * s;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_mxf8(d_tmem, sdesc_sw128(a_addr + kk * 32, 16, 1024),
                                  sdesc_sw128(b_addr + kk * 32, 16, 1024),
                                  idesc_mxf8_f32(128, BN, (uint32_t)kk), sfa, sfa + 4,
                                  (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(&empty[s]);
                }
                __syncwarp();
                if (++s == STAGES) { s = 0; ph ^= 1u; }
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
    } else if (warp >= 2 + NEPI) {
        // ------------------------------------------------ scale writers
        // per stage, the word of the stage's four scale codes of every A and B
        // row, in the layout the tensor cores read: each lane quadrant holds
        // all 128 rows of A and all BN rows of B, lane 32q + j at column
        // (first + c) holding row 32c + j (A at the stage's first four scale
        // columns, B at the next BN/32).  A stage's columns are rewritten once
        // its previous MMAs are done (empty), ahead of its codes.
        const int q = warp & 3;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        uint32_t s = 0, ph = 0, js = 0, phs = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            const int t = next_tile(i, false, 0xffffffffu);
            if (t < 0 || t >= total_tiles) break;
            const TileInfo ti = mx_tile<MODE>(p, t, mt_start, offs);
            for (int kb = 0; kb < ti.kb; ++kb) {
                if ((kb & 3) == 0 && !mbar_wait(&sffull[js], phs, wc)) { ok = false; break; }
                if (!mbar_wait(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
                tc_fence_after();
                const uint8_t *sa = sSf + js * SH::SF_SLOT;
                const uint8_t *sb = sa + kMxSfA;
                const uint32_t koff = (uint32_t)(kb & 3) * 4u;
                uint32_t wa[4], wb[BN / 32];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    wa[c] = *reinterpret_cast<const uint32_t *>(
                        sa + (uint32_t)(32 * c + lane) * kMxSfRow + koff);
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    wb[c] = *reinterpret_cast<const uint32_t *>(
                        sb + (uint32_t)(32 * c + lane) * kMxSfRow + koff);
                const uint32_t col = SH::SF_COL0 + SH::SF_COLS * s;
                tmem_st4(lane_base + col, wa[0], wa[1], wa[2], wa[3]);
#pragma unroll
                for (int c = 0; c < BN / 32; c += 4)
                    tmem_st4(lane_base + col + 4u + c, wb[c], wb[c + 1], wb[c + 2], wb[c + 3]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfready[s]);
                if ((kb & 3) == 3 || kb == ti.kb - 1) {
                    if (lane == 0) mbar_arrive(&sfempty[js]);
                    if (++js == kMxSfSlots) { js = 0; phs ^= 1u; }
                }
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..)
        // NEPI / 4 warps per TMEM lane quadrant, each taking an equal share of
        // the tile's columns
        const int q = warp & 3;   // TMEM lane quadrant this warp may read
        const int part = (warp - 2) >> 2;
        constexpr int NPART = NEPI / 4;
        const int r_local = q * 32 + lane;
        int it = 0;
        for (;; ++it) {
            const int t = next_tile(it, false, 0xffffffffu);
            if (t < 0 || t >= total_tiles) break;
            const TileInfo ti = mx_tile<MODE>(p, t, mt_start, offs);
            const uint32_t acc = NACC == 2 ? (it & 1) : 0;
            const uint32_t aph = NACC == 2 ? ((it >> 1) & 1) : (it & 1);
            if (!mbar_wait(&tfull[acc], aph, wc)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            const bool valid = r_local < ti.rows_valid;
            const int row = ti.row0 + r_local;
            if constexpr (MODE == MX_FFN1) {
                constexpr int HC = BN / 2 / NPART;   // h columns of this warp
#pragma unroll 1
                for (int c = part * HC; c < (part + 1) * HC; c += 32) {
                    uint32_t rg[32], ru[32];
                    tmem_ld32(tb + c, rg);
                    tmem_ld32(tb + BN / 2 + c, ru);
                    tmem_wait_ld();
                    if (valid) {
                        float hv[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            hv[j] = swiglu_clamped(__uint_as_float(rg[j]),
                                                        __uint_as_float(ru[j]), p.clamp);
                        uint32_t w[8];
                        const uint32_t code = mx_quantize_block(hv, w);
                        const int col = ti.nt * (BN / 2) + c;
                        uint8_t *dst = p.hq + (size_t)row * p.I + col;
                        st_global_v4(dst, w[0], w[1], w[2], w[3]);
                        st_global_v4(dst + 16, w[4], w[5], w[6], w[7]);
                        p.hsf[(size_t)row * p.h_pitch + col / 32] = (uint8_t)code;
                        if (p.gu_out) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                st_global_v4(p.gu_out + gu_offset(row, col + j, p.I), rg[j],
                                             rg[j + 1], rg[j + 2], rg[j + 3]);
                                st_global_v4(p.gu_out + gu_offset(row, p.I + col + j, p.I), ru[j],
                                             ru[j + 1], ru[j + 2], ru[j + 3]);
                            }
                        }
                    }
                }
            } else if constexpr (MODE == MX_DGRAD2) {
                constexpr int DC = BN / NPART;       // columns of dA of this warp
                // warps whose 32 rows all exist use TMA stores; the others direct ones
                const bool warp_full = q * 32 + 32 <= ti.rows_valid;
                uint8_t *stg = sEpi + (size_t)(warp - 2) * SH::EPI_WARP;
                float w = 1.0f;
                if (valid && p.row_w && row < p.w_rows) w = p.row_w[row];
                const float cl = p.clamp;
                float dw = 0.0f;
#pragma unroll 1
                for (int c = part * DC; c < (part + 1) * DC; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c, r);
                    tmem_wait_ld();
                    if (valid) {
                        const int col = ti.nt * BN + c;
                        // the forward's fp32 g, u and MX h~ of these 32 columns
                        float4 gv4[8], uv4[8];
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            gv4[q4] = *reinterpret_cast<const float4 *>(
                                p.gu_in + gu_offset(row, col + 4 * q4, p.I));
                            uv4[q4] = *reinterpret_cast<const float4 *>(
                                p.gu_in + gu_offset(row, p.I + col + 4 * q4, p.I));
                        }
                        const uint4 *hp =
                            reinterpret_cast<const uint4 *>(p.hq_in + (size_t)row * p.I + col);
                        const uint4 h0 = hp[0], h1 = hp[1];
                        const uint32_t hc[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                        const float hs = mx_scale(p.hsf_in[(size_t)row * p.h_pitch + col / 32]);
                        float *dg = reinterpret_cast<float *>(gv4);
                        float *du = reinterpret_cast<float *>(uv4);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            float h4[4];
                            e4m3x4_values(hc[j >> 2], h4);
                            const float g = dg[j], u = du[j];
                            const float dA = __uint_as_float(r[j]);
                            const float ht = h4[j & 3] * hs;
                            const float a = fminf(g, cl);
                            const float b = fminf(fmaxf(u, -cl), cl);
                            const float sg = sigmoid_fast(a);
                            const float dH = w * dA;
                            dw = fmaf(ht, dA, dw);
                            dg[j] = g <= cl ? dH * b * (sg + a * sg * (1.0f - sg)) : 0.0f;
                            du[j] = (u >= -cl && u <= cl) ? dH * (a * sg) : 0.0f;
                            r[j] = __float_as_uint(w * ht);
                        }
                        // five 32-column outputs of this thread's row, one at a time
                        // (few live registers): dg and du quantised along 2I (each 32
                        // columns one block), dg, du and w h~ in bf16.  A warp whose
                        // 32 rows all exist stages each as a 32 x 32 block in shared
                        // memory and writes it with one TMA store; a ragged warp must
                        // not write past its group's rows and stores directly.
                        const uint32_t b0 = smem_u32(stg);
                        if (warp_full) {
                            if (lane == 0) bulk_wait_group_read<0>();   // staging free again
                            __syncwarp();
                        }
                        uint8_t *sd = p.dgusf + (size_t)row * p.dgu_pitch;
                        auto emit_codes = [&](const float *v, int c, uint32_t soff) {
                            uint32_t wq[8];
                            sd[c / 32] = (uint8_t)mx_quantize_block(
                                *reinterpret_cast<const float(*)[32]>(v), wq);
                            if (warp_full) {
                                const uint32_t a = b0 + soff + (uint32_t)lane * 32u;
                                st_shared_v4(a, wq[0], wq[1], wq[2], wq[3]);
                                st_shared_v4(a + 16u, wq[4], wq[5], wq[6], wq[7]);
                            } else {
                                uint8_t *qd = p.dguq + (size_t)row * 2 * p.I + c;
                                st_global_v4(qd, wq[0], wq[1], wq[2], wq[3]);
                                st_global_v4(qd + 16, wq[4], wq[5], wq[6], wq[7]);
                            }
                        };
                        auto emit_bf16 = [&](const float *v, uint16_t *gdst, uint32_t soff) {
                            const uint32_t sw2 = (uint32_t)((lane >> 1) & 3);
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) {
                                const uint32_t x0 = pack_bf16x2(v[8 * jj], v[8 * jj + 1]);
                                const uint32_t x1 = pack_bf16x2(v[8 * jj + 2], v[8 * jj + 3]);
                                const uint32_t x2 = pack_bf16x2(v[8 * jj + 4], v[8 * jj + 5]);
                                const uint32_t x3 = pack_bf16x2(v[8 * jj + 6], v[8 * jj + 7]);
                                if (warp_full)
                                    st_shared_v4(b0 + soff + (uint32_t)lane * 64u +
                                                     ((((uint32_t)jj) ^ sw2) << 4),
                                                 x0, x1, x2, x3);
                                else
                                    st_global_v4(gdst + 8 * jj, x0, x1, x2, x3);
                            }
                        };
                        emit_codes(dg, col, 6144u);
                        emit_codes(du, p.I + col, 7168u);
                        uint16_t *dgd = p.dgu + (size_t)row * 2 * p.I + col;
                        emit_bf16(dg, dgd, 0u);
                        emit_bf16(du, dgd + p.I, 2048u);
                        emit_bf16(reinterpret_cast<const float *>(r), p.hw + (size_t)row * p.I + col,
                                  4096u);
                        if (warp_full) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int wrow = ti.row0 + q * 32;
                                tma_store_2d(&p.tmO, stg, col, wrow);
                                tma_store_2d(&p.tmO, stg + 2048, p.I + col, wrow);
                                tma_store_2d(&p.tmO2, stg + 4096, col, wrow);
                                tma_store_2d(&p.tmOQ, stg + 6144, col, wrow);
                                tma_store_2d(&p.tmOQ, stg + 7168, p.I + col, wrow);
                                bulk_commit_group();
                            }
                        }
                    }
                }
                // one partial of <h~, dA> per (row, column tile, warp part)
                if (valid) p.dw_part[((size_t)row * p.n_tiles + ti.nt) * NPART + part] = dw;
            } else if constexpr (MODE == MX_WGRAD) {
                // fp32 blocks of 32 rows x 32 columns through shared memory
                // (128-byte swizzle), one TMA store each; a group without rows
                // gets zeros (its accumulator was never written)
                constexpr int WC = BN / NPART;
                uint8_t *stg0 = sEpi + (size_t)(warp - 2) * 4096 * kMxWgradStageBufs;
                const uint32_t sw = (uint32_t)(lane & 7);
                const bool has_k = ti.kb > 0;
#pragma unroll 1
                for (int c = part * WC; c < (part + 1) * WC; c += 32) {
                    uint8_t *stg = stg0 + (kMxWgradStageBufs == 2 ? ((c >> 5) & 1) * 4096 : 0);
                    const uint32_t row_addr = smem_u32(stg) + (uint32_t)lane * 128u;
                    uint32_t r[32];
                    if (has_k) {
                        tmem_ld32(tb + c, r);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    // the store that last read this staging block is done with it
                    if (lane == 0) {
                        if constexpr (kMxWgradStageBufs == 2) bulk_wait_group_read<1>();
                        else bulk_wait_group_read<0>();
                    }
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(row_addr + ((((uint32_t)j) ^ sw) << 4), r[4 * j], r[4 * j + 1],
                                     r[4 * j + 2], r[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tmOQ, stg, ti.nt * BN + c, ti.g * p.M + ti.m0 + q * 32);
                        bulk_commit_group();
                    }
                }
            } else {
                constexpr int YC = BN / NPART;       // output columns of this warp
                float w = 1.0f;
                if (valid && p.row_w && row < p.w_rows) w = p.row_w[row];
#pragma unroll 1
                for (int c = part * YC; c < (part + 1) * YC; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c, r);
                    tmem_wait_ld();
                    if (valid) {
                        uint16_t *dst = p.y + (size_t)row * p.N + ti.nt * BN + c;
#pragma unroll
                        for (int j = 0; j < 32; j += 8)
                            st_global_v4(dst + j,
                                         pack_bf16x2(w * __uint_as_float(r[j]),
                                                     w * __uint_as_float(r[j + 1])),
                                         pack_bf16x2(w * __uint_as_float(r[j + 2]),
                                                     w * __uint_as_float(r[j + 3])),
                                         pack_bf16x2(w * __uint_as_float(r[j + 4]),
                                                     w * __uint_as_float(r[j + 5])),
                                         pack_bf16x2(w * __uint_as_float(r[j + 6]),
                                                     w * __uint_as_float(r[j + 7])));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
        // the TMA stores must have left shared memory (and landed) before exit
        if ((MODE == MX_DGRAD2 || MODE == MX_WGRAD) && lane == 0) bulk_wait_group_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kMxTmemCols);
}

template <int MODE, int BN>
moe_status launch_mx(MxParams &p, int max_tiles, cudaStream_t st) {
    using SH = MxShape<MODE, BN>;
    auto kern = moe_mx_gemm_kernel<MODE, BN>;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mx_smem_bytes<MODE, BN>(kMaxGroups)) != cudaSuccess)
            return MOE_ERR_CUDA;
        attr_set[dev] = true;
    }
    if (max_tiles <= 0) return MOE_OK;
    p.status = device_status_ptr();
    if (!p.status) return MOE_ERR_CUDA;
    if (p.wait_limit <= 0) p.wait_limit = kWaitLimitCycles;
    const int grid = max_tiles < num_sms() ? max_tiles : num_sms();
    kern<<<grid, SH::THREADS, mx_smem_bytes<MODE, BN>(p.G), st>>>(p);
    return cuda_status(cudaGetLastError());
}

}  // namespace

// 256-wide tiles (one accumulator) when the groups hold many rows, where the
// MMAs set the pace; 128-wide ones (two accumulators) otherwise.
static int mx_bn(int max_rows, int G) { return (long long)max_rows >= 1024LL * G ? 256 : 128; }

moe_status launch_mx_ffn1(const uint8_t *xq, const uint8_t *xsf, const int32_t *offsets, int G,
                          int max_rows, const uint8_t *W13q, const uint8_t *W13sf, int d, int I,
                          float clamp, uint8_t *hq, uint8_t *hsf, float *gu_save,
                          cudaStream_t st) {
    if (d % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    MxParams p;
    std::memset(&p, 0, sizeof p);
    const int BN = mx_bn(max_rows, G);
    const int sfd = mx_sf_pitch(d);
    const uint64_t brows = (uint64_t)G * 2 * I;
    if (!encode_tmap_u8_2d(&p.tmA, xq, d, max_rows, d, 128, 128, 128) ||
        !encode_tmap_u8_2d(&p.tmB, W13q, d, brows, d, 128, BN / 2, 128) ||
        !encode_tmap_u8_2d(&p.tmSA, xsf, sfd, max_rows, sfd, 16, 128, 0) ||
        !encode_tmap_u8_2d(&p.tmSB, W13sf, sfd, brows, sfd, 16, BN / 2, 0))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = I / (BN / 2);
    p.k_blocks = d / 128;
    p.b_rows_per_group = 2 * I;
    p.I = I;
    p.clamp = clamp;
    p.hq = hq;
    p.hsf = hsf;
    p.h_pitch = mx_sf_pitch(I);
    p.gu_out = gu_save;
    const int tiles = row_tile_bound(max_rows, G) * p.n_tiles;
    return BN == 256 ? launch_mx<MX_FFN1, 256>(p, tiles, st) : launch_mx<MX_FFN1, 128>(p, tiles, st);
}

moe_status launch_mx_ffn2(const uint8_t *hq, const uint8_t *hsf, const int32_t *offsets, int G,
                          int max_rows, const uint8_t *W2q, const uint8_t *W2sf,
                          const float *row_w, int S, int d, int I, uint16_t *y, cudaStream_t st) {
    if (d % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    MxParams p;
    std::memset(&p, 0, sizeof p);
    const int BN = mx_bn(max_rows, G);
    const int sfi = mx_sf_pitch(I);
    const uint64_t brows = (uint64_t)G * d;
    if (!encode_tmap_u8_2d(&p.tmA, hq, I, max_rows, I, 128, 128, 128) ||
        !encode_tmap_u8_2d(&p.tmB, W2q, I, brows, I, 128, BN, 128) ||
        !encode_tmap_u8_2d(&p.tmSA, hsf, sfi, max_rows, sfi, 16, 128, 0) ||
        !encode_tmap_u8_2d(&p.tmSB, W2sf, sfi, brows, sfi, 16, BN, 0))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = d / BN;
    p.k_blocks = I / 128;
    p.b_rows_per_group = d;
    p.I = I;
    p.N = d;
    p.y = y;
    p.row_w = row_w;
    p.w_rows = S;
    const int tiles = row_tile_bound(max_rows, G) * p.n_tiles;
    return BN == 256 ? launch_mx<MX_FFN2, 256>(p, tiles, st) : launch_mx<MX_FFN2, 128>(p, tiles, st);
}

moe_status launch_mx_dgrad2(const uint8_t *dYq, const uint8_t *dYsf, const int32_t *offsets, int G,
                            int max_rows, const uint8_t *W2tq, const uint8_t *W2tsf,
                            const float *gu, const uint8_t *hq, const uint8_t *hsf,
                            const float *row_w, int S, int d, int I, float clamp, uint16_t *dGU,
                            uint8_t *dGUq, uint8_t *dGUsf, uint16_t *hw, float *dw_part,
                            int *n_part, int *tile_counter, cudaStream_t st) {
    if (d % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    constexpr int BN = 128;   // two accumulators: a tile's epilogue overlaps the next's MMAs
    MxParams p;
    std::memset(&p, 0, sizeof p);
    // tiles handed out at run time from a counter that starts at 0
    if (!tile_counter) return MOE_ERR_INVALID_ARG;
    if (cudaMemsetAsync(tile_counter, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    p.tile_counter = tile_counter;
    const int sfd = mx_sf_pitch(d);
    const uint64_t brows = (uint64_t)G * I;
    if (!encode_tmap_u8_2d(&p.tmA, dYq, d, max_rows, d, 128, 128, 128) ||
        !encode_tmap_u8_2d(&p.tmB, W2tq, d, brows, d, 128, BN, 128) ||
        !encode_tmap_u8_2d(&p.tmSA, dYsf, sfd, max_rows, sfd, 16, 128, 0) ||
        !encode_tmap_u8_2d(&p.tmSB, W2tsf, sfd, brows, sfd, 16, BN, 0) ||
        !encode_tmap_bf16_2d_sw64(&p.tmO, dGU, 2 * I, max_rows, (uint64_t)4 * I, 32, 32) ||
        !encode_tmap_bf16_2d_sw64(&p.tmO2, hw, I, max_rows, (uint64_t)2 * I, 32, 32) ||
        !encode_tmap_u8_2d(&p.tmOQ, dGUq, 2 * I, max_rows, 2 * I, 32, 32, 0))
        return MOE_ERR_CUDA;
    p.offsets = offsets;
    p.G = G;
    p.n_tiles = I / BN;
    p.k_blocks = d / 128;
    p.b_rows_per_group = I;
    p.I = I;
    p.clamp = clamp;
    p.row_w = row_w;
    p.w_rows = S;
    p.gu_in = gu;
    p.hq_in = hq;
    p.hsf_in = hsf;
    p.h_pitch = mx_sf_pitch(I);
    p.dgu = dGU;
    p.dguq = dGUq;
    p.dgusf = dGUsf;
    p.dgu_pitch = mx_sf_pitch(2 * I);
    p.hw = hw;
    p.dw_part = dw_part;
    if (n_part) *n_part = mx_dgrad2_n_part(I);
    const int tiles = row_tile_bound(max_rows, G) * p.n_tiles;
    return launch_mx<MX_DGRAD2, BN>(p, tiles, st);
}

// One CTA, a thread per group (G <= 1025): korder, the groups in order of
// decreasing padded rows (ties by index), and the tile counter set to 0.
__global__ void __launch_bounds__(1024) mx_wgrad_order_kernel(const int32_t *kofs, int G,
                                                             int32_t *korder, int *counter) {
    __shared__ int32_t rows_s[1025];
    if (threadIdx.x == 0) *counter = 0;
    for (int g = threadIdx.x; g < G; g += blockDim.x) rows_s[g] = kofs[g + 1] - kofs[g];
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const int rg = rows_s[g];
        int rank = 0;
        for (int h = 0; h < G; ++h) {
            const int rh = rows_s[h];
            rank += (rh > rg || (rh == rg && h < g)) ? 1 : 0;
        }
        korder[rank] = g;
    }
}

moe_status launch_mx_wgrad(const uint8_t *At, const uint8_t *Atsf, const uint8_t *Bt,
                           const uint8_t *Btsf, const int32_t *kofs, const int32_t *sofs, int G,
                           int M, int N, int k_chunks, int sf_slots, float *dW, int32_t *korder,
                           int *tile_counter, cudaStream_t st) {
    if (M % 128 != 0 || N % 128 != 0 || k_chunks < 1 || sf_slots < 1) return MOE_ERR_UNSUPPORTED;
    if (G < 1 || G > 1025 || !korder || !tile_counter) return MOE_ERR_INVALID_ARG;
    constexpr int BN = 128;
    MxParams p;
    std::memset(&p, 0, sizeof p);
    // longest contraction first, tiles handed out at run time
    mx_wgrad_order_kernel<<<1, 1024, 0, st>>>(kofs, G, korder, tile_counter);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    p.korder = korder;
    p.tile_counter = tile_counter;
    // K-chunk-major operands: [chunks x rows, 128 codes] and [slots x rows, 16 scale codes]
    if (!encode_tmap_u8_2d(&p.tmA, At, 128, (uint64_t)k_chunks * M, 128, 128, 128, 128) ||
        !encode_tmap_u8_2d(&p.tmB, Bt, 128, (uint64_t)k_chunks * N, 128, 128, BN, 128) ||
        !encode_tmap_u8_2d(&p.tmSA, Atsf, 16, (uint64_t)sf_slots * M, 16, 16, 128, 0) ||
        !encode_tmap_u8_2d(&p.tmSB, Btsf, 16, (uint64_t)sf_slots * N, 16, 16, BN, 0) ||
        !encode_tmap_f32_2d(&p.tmOQ, dW, N, (uint64_t)G * M, (uint64_t)N * 4, 32, 32))
        return MOE_ERR_CUDA;
    p.offsets = kofs;
    p.sofs = sofs;
    p.G = G;
    p.M = M;
    p.N = N;
    p.n_tiles = N / BN;
    p.b_rows_per_group = 0;
    return launch_mx<MX_WGRAD, BN>(p, G * (M / 128) * (N / BN), st);
}

int mx_dgrad2_n_part(int I) { return I / 128 * (MxShape<MX_DGRAD2, 128>::NEPI / 4); }

}  // namespace moe

// gemm_kernel.cuh -- persistent tcgen05 grouped GEMM for the expert matmuls.
//
// One CTA per SM (or a 2-SM pair per SM pair), 2 + NEPI warps:
//   warp 0      TMA producer (one elected thread): A and B tiles of 64 K
//               elements per stage into 128-byte-swizzled shared memory.
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma (M = 128, N = BN,
//               K = 16) from shared-memory descriptors into a fp32
//               accumulator in TMEM; two accumulators so that the epilogue of
//               one tile overlaps the main loop of the next.
//   warps 2..   epilogue (4 warps, 8 for dgrad 2): tcgen05.ld of the
//               accumulator (thread = row), mode-specific arithmetic, direct
//               global stores or shared-memory staging (TMA stores for dgrad
//               2, a transpose to coalesced stores for the weight gradients).
//
// Tiles are 128 rows x BN columns.  Three tile spaces:
//   dense        (GM_GATE)   rows of A in order;
//   row-grouped  (FFN1/FFN2/DGRAD2/DGRAD1) rows of A partitioned into groups
//                by offsets[]; each group's rows are tiled by 128 (the last
//                tile of a group is ragged and masked at the store), and the
//                group selects its expert's weights;
//   K-grouped    (GM_WGRAD) the contraction runs over each group's rows
//                (ragged K, zero rows -> zero output), output [G, M, N].
// GM_FFN12 runs the row-grouped tiles of expert GEMM 1 and then those of
// expert GEMM 2 in one launch: a GEMM-2 row tile's producer waits (bounded)
// until every epilogue warp of the GEMM-1 tiles of that row tile has
// released its h rows through a counter.
// The forward GEMMs and dgrad 1, whose tiles all cost the same, take them in
// a static round robin (tile = cluster + i * clusters); dgrad 2 and the weight
// gradients take them at run time from a global counter (see DYN in the
// kernel).  Either way each output tile is computed whole by one CTA (or
// pair) in a fixed contraction order, so the results are deterministic.
//
// CL = 2 (row-grouped and K-grouped modes): clusters of two CTAs run 2-SM
// MMAs (tcgen05.mma.cta_group::2, M = 256).  The pair computes two 128-row
// tiles of the same group and column tile; CTA r loads its own 128 rows of A
// and half of the B tile (columns [r BN/2, (r+1) BN/2)) with plain TMA
// copies, so each CTA reads half the B bytes per MMA that a lone CTA does and
// more operand stages fit.  The odd CTA's copies complete on the even CTA's
// barrier of the stage (cta_group::2 TMA), so the even CTA issues the MMAs
// once both CTAs' halves have landed, and releases stages and accumulators to
// both CTAs with one commit; every epilogue warp of the pair hands its drained
// accumulator back to the even CTA.
//
// K-grouped tiles whose rows end inside a 16-row MMA step: the producer loads
// that k-block's A through a copy of A's tensor map whose rows end at the
// group's last row (built on the device before the launch), so the rows past
// the group's end land as zeros (TMA fill) and no thread has to clear them.
//
// Every wait is bounded (moe_ptx.cuh): on a timeout the CTA records
// MOE_ERR_TIMEOUT, drains its own TMA copies and MMAs, frees TMEM and exits.
#pragma once

#include "moe_ptx.cuh"

namespace moe {

constexpr int kStageBudget = 192 * 1024;

struct GemmParams {
    CUtensorMap tmA;
    CUtensorMap tmB;
    CUtensorMap tmO;         // GM_WGRAD: fp32 output [G*M, N]; GM_DGRAD2: dGU [rows, 2I] bf16
    CUtensorMap tmO2;        // GM_DGRAD2: w h [rows, I] bf16 (boxes of 32 x 32)
    const int32_t *offsets;  // [G+1] group row offsets (grouped modes)
    // GM_WGRAD: per group, tmA with rows ending at the group's last row; the
    // groups in order of decreasing rows (ties by index); the tiles handed out
    // so far (zero before the launch)
    const CUtensorMap *tail_maps;
    const int32_t *korder;
    int *tile_counter;
    int G;
    int rows;                // GM_GATE: rows of A
    int n_tiles;             // column tiles per row tile
    int m_tiles;             // GM_WGRAD: M / 128
    int k_blocks;            // fixed-K modes: K / 64
    int N;                   // output columns (row pitch of the main output)
    int M;                   // GM_WGRAD: output rows per group
    int b_rows_per_group;    // rows of the flat weight matrix per group
    int I;                   // intermediate size (FFN1 / DGRAD2)
    float clamp;
    void *out;               // main output
    void *out2;              // FFN1: fp32 g|u save, gu_offset layout (nullable); DGRAD2: dGU
    void *out3;              // DGRAD2: w h
    float *out4;             // DGRAD2: dw partials [rows, n_tiles * 2]
    const float *row_w;      // FFN2 / DGRAD2 routing weight of rows < w_rows
    int w_rows;
    const float *gu_in;      // DGRAD2: saved fp32 g|u (gu_offset layout)
    const float *col_add;    // GM_GATE: per-column offset (nullable)
    // GM_FFN12: the GEMM-2 phase (A = h through tmO, B = W2 through tmO2,
    // y to out3) and the per-row-tile counters of finished GEMM-1 warps
    int n_tiles2, k_blocks2, b_rows2;
    int *ready;
    int ready_target;
    int stall_rt;            // GM_FFN12 test hook: this row tile never becomes ready (-1: none)
    int *status;
    long long wait_limit;
};

template <int MODE>
struct ModeTraits {
    // epilogue warps: two per TMEM lane quadrant (each drains half the
    // columns) for the heavy SwiGLU-backward epilogue of dgrad 2, one
    // otherwise (the weight gradients gain more from a fourth operand stage
    // than from a wider epilogue)
    static constexpr int NEPI = (MODE == GM_DGRAD2) ? 8 : 4;
    static constexpr int THREADS = 64 + 32 * NEPI;
    static constexpr bool A_MN = (MODE == GM_WGRAD);
    static constexpr bool B_MN = (MODE == GM_DGRAD2 || MODE == GM_DGRAD1 || MODE == GM_WGRAD);
    static constexpr bool DENSE = (MODE == GM_GATE);
    static constexpr bool KGROUP = (MODE == GM_WGRAD);
    static constexpr bool ROWGROUP = !DENSE && !KGROUP;
};

// Epilogue staging, per epilogue warp:
//   GM_WGRAD   one 32 x 32 fp32 block (4 KB): written one row per lane
//              (128-byte swizzle, conflict-free), read back four rows per
//              instruction and stored as full 128-byte lines with st.global.
//              The staging is free again as soon as it has been read back, so
//              one 4 KB buffer per warp keeps the SM's store path busy (TMA
//              stores would hold it until the copy engine has read it: with
//              one buffer per warp they reach ~20 B/cycle per SM, against the
//              ~30 that plain coalesced stores reach).
//   GM_DGRAD2  one 32 x 32 bf16 block (2 KB, 64-byte swizzle) that dg, du and
//              w h pass through in turn on their way to TMA stores: the
//              smaller staging leaves room for a fourth operand stage, which
//              the contraction over d = 4096 needs more than the epilogue
//              needs three blocks in flight.
constexpr int kEpiWarpBytes = 4096;
constexpr int kEpiWarpBytesDgrad2 = 2048;
// Barriers, TMEM base, abort flag and tile-index ring of one CTA.
constexpr int kBarBlockBytes = 512;
// Run-time tile order (dgrad 2, the weight gradients): slots of the ring that
// hands each tile index from the scheduling thread to the other roles.
constexpr int kSchedSlots = 8;
// Weight gradients' L2 policies: bit 0 operand loads evict-last, bit 1 the
// fp32 output stores evict-first.
constexpr int kWgradL2Hints = 3;
// Operand stages plus epilogue staging of the staged-epilogue modes.
constexpr int kStoreModeBudget = 216 * 1024;

template <int BN, int MODE, int CL = 1>
struct TileShape {
    static constexpr bool TMA_STORE = (MODE == GM_DGRAD2);
    static constexpr bool STAGED_EPI = (MODE == GM_WGRAD || MODE == GM_DGRAD2);
    static constexpr int A_BYTES = 128 * 64 * 2;
    static constexpr int B_BYTES = (BN / CL) * 64 * 2;   // this CTA's share of the B tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BYTES =
        MODE == GM_WGRAD    ? ModeTraits<MODE>::NEPI * kEpiWarpBytes
        : MODE == GM_DGRAD2 ? ModeTraits<MODE>::NEPI * kEpiWarpBytesDgrad2
                            : 0;
    static constexpr int STAGES =
        ((STAGED_EPI ? kStoreModeBudget : kStageBudget) - EPI_BYTES) / STAGE_BYTES;
    static constexpr uint32_t TMEM_COLS = 2 * BN;  // BN in {64, 128, 256}: a power of two
};

// Dynamic shared memory of one CTA for G groups.
template <int BN, int MODE, int CL = 1>
inline size_t gemm_smem_bytes(int G) {
    using TS = TileShape<BN, MODE, CL>;
    return 1024 + (size_t)TS::STAGES * TS::STAGE_BYTES + TS::EPI_BYTES + kBarBlockBytes +
           8 * (size_t)(G + 2);
}

struct TileInfo {
    int g;           // group
    int row0;        // first output / A row (row modes), 0 otherwise
    int rows_valid;  // rows of the tile that exist (row modes)
    int nt;          // column tile
    int m0;          // GM_WGRAD: first output row inside the group
    int krow0;       // GM_WGRAD: first contraction row
    int krows;       // GM_WGRAD: contraction rows
    int kb;          // k blocks of 64
    int phase;       // GM_FFN12: 0 = GEMM 1, 1 = GEMM 2
    int rt;          // row modes: index of the row tile (over all groups)
};

// Tile t of the schedule.  With CL = 2 (a 2-SM pair) t counts pairs of
// 128-row tiles of the same group and column tile, and `rank` picks the CTA's
// tile of the pair; a pair's second tile may lie past the group's rows
// (rows_valid <= 0: computed, never stored).
template <int MODE, int BN, int CL>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams &p, int t, const int *mt_start,
                                                const int *offs, int rank) {
    using MT = ModeTraits<MODE>;
    TileInfo ti;
    int tt = t, ntc = p.n_tiles;
    ti.phase = 0;
    if constexpr (MODE == GM_FFN12) {
        const int t1 = mt_start[p.G] * p.n_tiles;   // tiles of GEMM 1
        if (t >= t1) {
            tt = t - t1;
            ntc = p.n_tiles2;
            ti.phase = 1;
        }
    }
    ti.nt = tt % ntc;
    const int q = tt / ntc;
    ti.rt = q;
    ti.m0 = 0;
    ti.krow0 = 0;
    ti.krows = 0;
    if constexpr (MT::DENSE) {
        ti.g = 0;
        ti.row0 = (q * CL + rank) * 128;
        ti.rows_valid = min(128, p.rows - ti.row0);
        ti.kb = p.k_blocks;
    } else if constexpr (MT::ROWGROUP) {
        int lo = 0, hi = p.G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (mt_start[mid] <= q) lo = mid; else hi = mid - 1;
        }
        ti.g = lo;
        ti.row0 = offs[lo] + ((q - mt_start[lo]) * CL + rank) * 128;
        ti.rows_valid = min(128, offs[lo + 1] - ti.row0);
        ti.kb = ti.phase ? p.k_blocks2 : p.k_blocks;
    } else {
        // groups by decreasing rows (mt_start holds that order here): the
        // largest contractions first, the short ones last
        const int mp = p.m_tiles / CL;
        ti.g = mt_start[q / mp];
        ti.m0 = ((q % mp) * CL + rank) * 128;
        ti.row0 = 0;
        ti.rows_valid = 128;
        ti.krow0 = offs[ti.g];
        ti.krows = max(0, offs[ti.g + 1] - ti.krow0);
        ti.kb = (ti.krows + 63) >> 6;
    }
    return ti;
}

// K-grouped modes: the group's rows end inside the last 16-row MMA step of
// k-block kb of the tile (the rest of that step would be the next group's
// rows).
__device__ __forceinline__ bool kgroup_ragged(const TileInfo &ti, int kb) {
    const int valid = ti.krows - kb * 64;
    return valid < 64 && (valid & 15) != 0;
}

// The i-th tile of cluster cid (ncl clusters) in the static modes: round
// robin (their tiles all have the same length).
__device__ __forceinline__ int tile_at(int i, int cid, int ncl) { return i * ncl + cid; }

// Offset (in floats) of element (row, col) of the saved fp32 [g | u] buffer.
// Layout: blocks of 32 rows; inside a block, groups of 4 columns; inside a
// group, the 32 rows' 4 values back to back.  An epilogue warp owns 32
// consecutive rows (one per lane), so its 16-byte accesses to a column group
// cover one or two contiguous 512-byte runs instead of 32 scattered rows.
__device__ __forceinline__ size_t gu_offset(int row, int col, int I) {
    return ((size_t)(row >> 5) * (size_t)(I >> 1) + (size_t)(col >> 2)) * 128 +
           (size_t)(row & 31) * 4 + (size_t)(col & 3);
}

// sigmoid(a) with the fast exponential and division (a few ulp of fp32, far
// below the bf16 or E4M3 rounding of everything computed from it).
__device__ __forceinline__ float sigmoid_fast(float a) {
    return __fdividef(1.0f, 1.0f + __expf(-a));
}

// h = silu(min(g, c)) * clamp(u, -c, c).  The forward's epilogues and dgrad 2's
// recompute of h call this one function on the same fp32 g and u, so the two
// agree bit for bit.
__device__ __forceinline__ float swiglu_clamped(float g, float u, float c) {
    const float a = fminf(g, c);
    const float b = fminf(fmaxf(u, -c), c);
    return a * sigmoid_fast(a) * b;
}

// Epilogue of expert GEMM 1 (one thread = one row of the tile): the clamped
// SwiGLU of the accumulator's gate half (columns [0, BN/2)) and up half ->
// h (bf16), plus the fp32 g|u when it is saved for the backward.
template <int BN>
__device__ __forceinline__ void epi_swiglu(const GemmParams &p, const TileInfo &ti, uint32_t tb,
                                           bool valid, int row) {
    constexpr int BH = BN / 2;
    uint16_t *h = static_cast<uint16_t *>(p.out);
    float *gu = static_cast<float *>(p.out2);
#pragma unroll 1
    for (int c = 0; c < BH; c += 32) {
        uint32_t rg[32], ru[32];
        tmem_ld32(tb + c, rg);
        tmem_ld32(tb + BH + c, ru);
        tmem_wait_ld();
        if (valid) {
            const int col = ti.nt * BH + c;
            uint32_t hp[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                hp[j] = pack_bf16x2(
                    swiglu_clamped(__uint_as_float(rg[2 * j]), __uint_as_float(ru[2 * j]), p.clamp),
                    swiglu_clamped(__uint_as_float(rg[2 * j + 1]), __uint_as_float(ru[2 * j + 1]),
                                   p.clamp));
            if (h) {
                uint16_t *dst = h + (size_t)row * p.I + col;
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    st_global_v4(dst + 2 * j, hp[j], hp[j + 1], hp[j + 2], hp[j + 3]);
            }
            if (gu) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    st_global_v4(gu + gu_offset(row, col + j, p.I), rg[j], rg[j + 1], rg[j + 2],
                                 rg[j + 3]);
                    st_global_v4(gu + gu_offset(row, p.I + col + j, p.I), ru[j], ru[j + 1],
                                 ru[j + 2], ru[j + 3]);
                }
            }
        }
    }
}

// Epilogue of expert GEMM 2 and dgrad 1: the accumulator times w -> bf16
// columns [nt BN, (nt + 1) BN) of this thread's row of y (row pitch N).
template <int BN>
__device__ __forceinline__ void epi_bf16_scaled(uint16_t *y, int N, const TileInfo &ti, uint32_t tb,
                                                bool valid, int row, float w) {
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld32(tb + c, r);
        tmem_wait_ld();
        if (valid) {
            uint16_t *dst = y + (size_t)row * N + ti.nt * BN + c;
#pragma unroll
            for (int j = 0; j < 32; j += 8)
                st_global_v4(dst + j,
                             pack_bf16x2(w * __uint_as_float(r[j]), w * __uint_as_float(r[j + 1])),
                             pack_bf16x2(w * __uint_as_float(r[j + 2]), w * __uint_as_float(r[j + 3])),
                             pack_bf16x2(w * __uint_as_float(r[j + 4]), w * __uint_as_float(r[j + 5])),
                             pack_bf16x2(w * __uint_as_float(r[j + 6]), w * __uint_as_float(r[j + 7])));
        }
    }
}

// CL = 1: one CTA per tile.  CL = 2: a 2-SM pair per two tiles (see above).
template <int MODE, int BN, int CL>
__global__ void __launch_bounds__(ModeTraits<MODE>::THREADS, 1)
    moe_gemm_kernel(const __grid_constant__ GemmParams p) {
    using MT = ModeTraits<MODE>;
    static_assert(CL == 1 || CL == 2, "one CTA or a 2-SM pair");
    static_assert(CL == 1 || (BN >= 128 && !MT::DENSE && MODE != GM_FFN12),
                  "the pair form: row- or K-grouped modes, 64-column B boxes per CTA");
    using TS = TileShape<BN, MODE, CL>;
    constexpr int STAGES = TS::STAGES;
    // the barrier block (full and empty per stage, two tfull, two tempty,
    // done, sfull and sempty per ring slot, the TMEM base, the abort flag and
    // the ring) must fit the bytes the layout reserves
    static_assert((2 * STAGES + 5 + 2 * kSchedSlots) * 8 + 8 + 4 * kSchedSlots <= kBarBlockBytes,
                  "too many operand stages for the barrier block");
    constexpr uint32_t IDESC = idesc_bf16_f32(128 * CL, BN, MT::A_MN, MT::B_MN);
    // tiles handed out at run time through the ring (see below): the K-grouped
    // weight gradients and dgrad 2, whose clusters otherwise drift apart
    constexpr bool DYN = MT::KGROUP || MODE == GM_DGRAD2;

    extern __shared__ uint8_t smem_raw[];
    // aligned to 1024 B by pointer arithmetic on the shared array itself, so
    // that the compiler keeps every access derived from it in the shared
    // state space (LDS/STS, shared atomics) instead of generic addressing
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * TS::A_BYTES;
    uint8_t *sEpi = smem + STAGES * TS::STAGE_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(sEpi + TS::EPI_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    // K-grouped modes: ring of run-time tile indices (sched), filled by the
    // scheduling thread (sfull) and released by every other role (sempty)
    uint64_t *sfull = done + 1;
    uint64_t *sempty = sfull + kSchedSlots;
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(sempty + kSchedSlots);
    volatile int *abort_s = reinterpret_cast<volatile int *>(tmem_base_s + 1);
    volatile int *sched = abort_s + 1;
    int *offs = reinterpret_cast<int *>(smem + STAGES * TS::STAGE_BYTES + TS::EPI_BYTES +
                                        kBarBlockBytes);
    int *mt_start = offs + (p.G + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            // CL = 2: one arrival per epilogue warp of either CTA
            mbar_init(&tempty[a], CL == 1 ? 32 * MT::NEPI : 2 * MT::NEPI);
        }
        mbar_init(done, 1);
        for (int j = 0; j < kSchedSlots; ++j) {
            mbar_init(&sfull[j], 1);
            // readers: CL = 2 both issuers, the odd producer and every epilogue
            // warp of both CTAs; CL = 1 the issuer and the epilogue warps
            mbar_init(&sempty[j], CL == 2 ? 3 + 2 * MT::NEPI : 1 + MT::NEPI);
        }
        *abort_s = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(&p.tmB);
        if constexpr (TS::TMA_STORE || MODE == GM_FFN12) tma_prefetch_desc(&p.tmO);
        if constexpr (MODE == GM_FFN12) tma_prefetch_desc(&p.tmO2);
        if constexpr (MODE == GM_DGRAD2) tma_prefetch_desc(&p.tmO2);
    }
    if (warp == 1) {
        if constexpr (CL == 2) {
            tmem_alloc_pair(tmem_base_s, TS::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_base_s, TS::TMEM_COLS);
            tmem_relinquish();
        }
    }
    if constexpr (!MT::DENSE) {
        if (warp == 2) {
            // group offsets and (row modes) the exclusive prefix of 128-row tiles
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
                    mt = (mt + CL - 1) / CL;   // tiles, or pairs of tiles
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
            // K-grouped modes: the group order of the schedule in place of the
            // (unused) tile prefix
            if constexpr (MT::KGROUP)
                for (int g = lane; g < p.G; g += 32) mt_start[g] = p.korder[g];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the pair's commits and forwarded arrivals target both CTAs' barriers:
    // both must have initialised them first
    if constexpr (CL == 2) cluster_sync_all();
    const int rank = CL == 2 ? (int)cluster_ctarank() : 0;
    const int cid = blockIdx.x / CL;          // cluster index
    const int ncl = gridDim.x / CL;           // clusters in the grid

    const uint32_t tmem_base = *tmem_base_s;
    const WaitCtl wc{abort_s, p.status, p.wait_limit};
    int total_tiles;
    if constexpr (MT::DENSE) {
        total_tiles = ((((p.rows + 127) >> 7) + CL - 1) / CL) * p.n_tiles;
    } else if constexpr (MT::ROWGROUP) {
        total_tiles = mt_start[p.G] * (MODE == GM_FFN12 ? p.n_tiles + p.n_tiles2 : p.n_tiles);
    } else {
        total_tiles = p.G * (p.m_tiles / CL) * p.n_tiles;
    }

    // DYN modes hand the tiles out at run time, in tile order (K-grouped: the
    // group list, longest contraction first), from a global counter.  The tiles
    // in flight at any moment are then a window of about one tile per cluster,
    // so the tiles that share an expert's operand rows run together and find
    // them in L2.  Under a static round robin the clusters drifted apart (the
    // weight gradients' tile lengths differ from group to group; dgrad 2's
    // epilogue time varies) by thousands, or hundreds, of tiles, and those rows
    // were read from DRAM several times over.  The even CTA's producer takes
    // each index and passes it through the ring (sched) to every other role of
    // both CTAs; total_tiles marks the end.  Other modes deal tiles statically.
    auto sched_put = [&](int i) -> int {
        const int j = i % kSchedSlots;
        if (!mbar_wait(&sempty[j], ((uint32_t)(i / kSchedSlots) & 1u) ^ 1u, wc)) return -1;
        int t = atomicAdd(p.tile_counter, 1);
        if (t > total_tiles) t = total_tiles;
        sched[j] = t;
        if constexpr (CL == 2) {
            dsmem_st_u32(dsmem_map(const_cast<int *>(&sched[j]), 1), (uint32_t)t);
            mbar_arrive_remote(dsmem_map(&sfull[j], 1));
        }
        mbar_arrive(&sfull[j]);
        return t;
    };
    // a reader of slot i % kSchedSlots (mask: the lanes of the calling warp
    // that read it; lane 0 releases the slot once the index has been read)
    auto sched_get = [&](int i, uint32_t mask) -> int {
        const int j = i % kSchedSlots;
        const uint32_t sp = (uint32_t)(i / kSchedSlots) & 1u;
        const bool got = rank == 0 ? mbar_wait(&sfull[j], sp, wc) : mbar_wait_cluster(&sfull[j], sp, wc);
        if (!got) return -1;
        const int t = sched[j];
        __syncwarp(mask);
        // the arrival depends on the index read, so it cannot pass that read
        if (lane == 0 && t >= 0) {
            if (rank == 0) mbar_arrive(&sempty[j]);
            else mbar_arrive_remote_relaxed(dsmem_map(&sempty[j], 0));
        }
        return t;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_op = policy_evict_last();
            int last_par[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
            uint32_t s = 0, ph = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                int t;
                if constexpr (DYN) t = rank == 0 ? sched_put(i) : sched_get(i, 1u);
                else t = tile_at(i, cid, ncl);
                if (t < 0) { ok = false; break; }
                if (t >= total_tiles) break;
                const TileInfo ti = decode_tile<MODE, BN, CL>(p, t, mt_start, offs, rank);
                if constexpr (MODE == GM_FFN12) {
                    if (ti.phase == 1) {
                        // the h rows of this row tile: every epilogue warp of its
                        // GEMM-1 tiles has released them (earlier tiles of the
                        // static order, all on resident CTAs).  The writers
                        // fenced their stores into the async proxy before the
                        // release, so the copies below may read them at once.
                        const int target = p.ready_target + (ti.rt == p.stall_rt ? 1 : 0);
                        if (!wait_count_geq(p.ready + ti.rt, target, wc)) {
                            ok = false;
                            break;
                        }
                    }
                }
                for (int kb = 0; kb < ti.kb; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
                    // CL = 2: the even CTA's barrier takes both CTAs' halves of
                    // every stage
                    const bool to_even = CL == 2 && rank == 1;
                    uint32_t bar_even = 0;
                    if (to_even)
                        bar_even = dsmem_map(&full[s], 0);
                    else
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(CL * TS::STAGE_BYTES));
                    auto load = [&](void *dst, const CUtensorMap *tm, int c0, int c1) {
                        if constexpr (MT::KGROUP && (kWgradL2Hints & 1)) {
                            if (to_even) tma_load_2d_pairbar_hint(dst, tm, bar_even, c0, c1, pol_op);
                            else tma_load_2d_hint(dst, tm, &full[s], c0, c1, pol_op);
                        } else {
                            if (to_even) tma_load_2d_pairbar(dst, tm, bar_even, c0, c1);
                            else tma_load_2d(dst, tm, &full[s], c0, c1);
                        }
                    };
                    uint8_t *a_dst = sA + s * TS::A_BYTES;
                    uint8_t *b_dst = sB + s * TS::B_BYTES;
                    if constexpr (MT::A_MN) {
                        // a k-block whose last 16-row step reaches past the
                        // group: A through the group's own map, whose rows end
                        // at the group's last row, so the rows past it land as
                        // zeros (TMA fill) and nothing has to clear them
                        const CUtensorMap *ta = &p.tmA;
                        if (kgroup_ragged(ti, kb)) {
                            ta = p.tail_maps + ti.g;
                            fence_tmap_acquire(ta);
                        }
                        load(a_dst, ta, ti.m0, ti.krow0 + kb * 64);
                        load(a_dst + 8192, ta, ti.m0 + 64, ti.krow0 + kb * 64);
                    } else if (MODE == GM_FFN12 && ti.phase == 1) {
                        load(a_dst, &p.tmO, kb * 64, ti.row0);
                    } else {
                        load(a_dst, &p.tmA, kb * 64, ti.row0);
                    }
                    if constexpr (CL == 1) {
                        if constexpr (MODE == GM_FFN12) {
                            if (ti.phase == 0) {
                                const int r = ti.g * p.b_rows_per_group + ti.nt * (BN / 2);
                                load(b_dst, &p.tmB, kb * 64, r);
                                load(b_dst + (BN / 2) * 128, &p.tmB, kb * 64,
                                            r + p.I);
                            } else {
                                load(b_dst, &p.tmO2, kb * 64,
                                            ti.g * p.b_rows2 + ti.nt * BN);
                            }
                        } else if constexpr (MODE == GM_GATE) {
                            load(b_dst, &p.tmB, kb * 64, ti.nt * BN);
                        } else if constexpr (MODE == GM_FFN1) {
                            const int r = ti.g * p.b_rows_per_group + ti.nt * (BN / 2);
                            load(b_dst, &p.tmB, kb * 64, r);
                            load(b_dst + (BN / 2) * 128, &p.tmB, kb * 64,
                                        r + p.I);
                        } else if constexpr (MODE == GM_FFN2) {
                            load(b_dst, &p.tmB, kb * 64,
                                        ti.g * p.b_rows_per_group + ti.nt * BN);
                        } else {
                            // MN-major B: BN/64 boxes of 64 columns x 64 contraction rows
                            const int krow = MT::KGROUP ? ti.krow0 + kb * 64
                                                        : ti.g * p.b_rows_per_group + kb * 64;
#pragma unroll
                            for (int j = 0; j < BN / 64; ++j)
                                load(b_dst + j * 8192, &p.tmB, ti.nt * BN + 64 * j, krow);
                        }
                    } else {
                        // 2-SM pair: this CTA's half of the B tile, into its own stage
                        if constexpr (MODE == GM_FFN1) {
                            // rank 0: the gate rows, rank 1: the matching up rows
                            const int r = ti.g * p.b_rows_per_group + ti.nt * (BN / 2);
                            load(b_dst, &p.tmB, kb * 64, r + rank * p.I);
                        } else if constexpr (MODE == GM_FFN2) {
                            load(b_dst, &p.tmB, kb * 64,
                                        ti.g * p.b_rows_per_group + ti.nt * BN + rank * (BN / 2));
                        } else {
                            // MN-major B: BN/128 boxes of 64 columns x 64 contraction rows
                            const int krow = MT::KGROUP ? ti.krow0 + kb * 64
                                                        : ti.g * p.b_rows_per_group + kb * 64;
#pragma unroll
                            for (int j = 0; j < BN / 128; ++j)
                                load(b_dst + j * 8192, &p.tmB, ti.nt * BN + rank * (BN / 2) + 64 * j, krow);
                        }
                    }
                    last_par[s] = (int)ph;
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok && CL == 2 && rank == 1) {
                // this CTA's copies complete on the even CTA's barriers, which it
                // cannot wait on: give those still in flight time to land (a
                // copy takes microseconds; this waits about a millisecond)
                const long long t0 = clock64();
                while (clock64() - t0 < (1LL << 21)) __nanosleep(1000);
            } else if (!ok) {
                // drain the copies still in flight before the CTA exits
                for (int i = 0; i < STAGES; ++i)
                    if (last_par[i] >= 0)
                        mbar_wait_teardown(&full[i], (uint32_t)last_par[i], p.wait_limit);
            } else if constexpr (CL == 2) {
                // every release of a stage (the even CTA's commits) must have
                // landed in our barriers before the CTA may exit
                for (int i = 0; i < STAGES; ++i)
                    if (last_par[i] >= 0)
                        mbar_wait_teardown(&empty[i], (uint32_t)last_par[i], p.wait_limit);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // CL = 2: the even CTA issues the pair's MMAs (the odd CTA's warp only
        // keeps its stage count).
        const bool issuer = CL == 1 || rank == 0;
        uint32_t s = 0, ph = 0;
        int it = 0;
        bool ok = true;
        bool issued = false;
        // ragged contraction: only the 16-row MMA steps that hold rows of this
        // group run; A's rows of the last one past the group's end landed as
        // zeros (the producer loads them through the group's own tensor map).
        // B's rows there are finite data or TMA zero fill, so they add nothing.
        for (; ok; ++it) {
            int t;
            if constexpr (DYN) t = sched_get(it, 0xffffffffu);
            else t = tile_at(it, cid, ncl);
            if (t < 0) { ok = false; break; }
            if (t >= total_tiles) break;
            const TileInfo ti = decode_tile<MODE, BN, CL>(p, t, mt_start, offs, rank);
            const uint32_t acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (issuer) {
                const bool got = CL == 2 ? mbar_wait_cluster(&tempty[acc], aph ^ 1u, wc)
                                         : mbar_wait(&tempty[acc], aph ^ 1u, wc);
                if (!got) { ok = false; break; }
                tc_fence_after();
            }
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < ti.kb; ++kb) {
                const int valid = MT::KGROUP ? ti.krows - kb * 64 : 64;
                if constexpr (CL == 2) {
                    if (rank == 1) {
                        if (++s == STAGES) { s = 0; ph ^= 1u; }
                        continue;
                    }
                }
                if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + s * TS::A_BYTES);
                const uint32_t b_addr = smem_u32(sB + s * TS::B_BYTES);
                const int n_kk = valid < 64 ? (valid + 15) >> 4 : 4;

                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (kk >= n_kk) break;
                        const uint64_t ad = MT::A_MN ? sdesc_sw128(a_addr + kk * 2048, 8192, 1024)
                                                     : sdesc_sw128(a_addr + kk * 32, 16, 1024);
                        const uint64_t bd = MT::B_MN ? sdesc_sw128(b_addr + kk * 2048, 8192, 1024)
                                                     : sdesc_sw128(b_addr + kk * 32, 16, 1024);
                        if constexpr (CL == 2)
                            umma_bf16_pair(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                        else
                            umma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    if constexpr (CL == 2) umma_commit_pair(&empty[s], 0x3);
                    else umma_commit(&empty[s]);
                }
                issued = true;
                __syncwarp();
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
            if (issuer) {
                if (lane == 0) {
                    if constexpr (CL == 2) umma_commit_pair(&tfull[acc], 0x3);
                    else umma_commit(&tfull[acc]);
                }
                __syncwarp();
            }
        }
        if (issuer && (CL == 2 ? issued : !ok)) {
            // every MMA this thread issued must finish before TMEM is freed (and,
            // for a pair, before either CTA's operand stages go away)
            if (lane == 0) {
                if constexpr (CL == 2) umma_commit_pair(done, 0x1);
                else umma_commit(done);
            }
            __syncwarp();
            mbar_wait_teardown(done, 0, p.wait_limit);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..)
        const int q = warp & 3;           // TMEM lane quadrant this warp may read
        const int ew = warp - 2;          // epilogue warp index
        const int r_local = q * 32 + lane;
        int it = 0;
        for (;; ++it) {
            int t;
            if constexpr (DYN) t = sched_get(it, 0xffffffffu);
            else t = tile_at(it, cid, ncl);
            if (t < 0 || t >= total_tiles) break;
            const TileInfo ti = decode_tile<MODE, BN, CL>(p, t, mt_start, offs, rank);
            const uint32_t acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(&tfull[acc], aph, wc)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            const bool valid = r_local < ti.rows_valid;
            const int row = ti.row0 + r_local;

            if constexpr (MODE == GM_GATE) {
                float *out = static_cast<float *>(p.out);
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c, r);
                    tmem_wait_ld();
                    const int col = ti.nt * BN + c;
                    if (valid && col < p.N) {
                        float *dst = out + (size_t)row * p.N + col;
                        if (col + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                float v[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    v[e] = __uint_as_float(r[j + e]) +
                                           (p.col_add ? p.col_add[col + j + e] : 0.0f);
                                st_global_v4(dst + j, __float_as_uint(v[0]), __float_as_uint(v[1]),
                                             __float_as_uint(v[2]), __float_as_uint(v[3]));
                            }
                        } else {
                            for (int j = 0; j < 32 && col + j < p.N; ++j)
                                dst[j] = __uint_as_float(r[j]) +
                                         (p.col_add ? p.col_add[col + j] : 0.0f);
                        }
                    }
                }
            } else if constexpr (MODE == GM_FFN1) {
                epi_swiglu<BN>(p, ti, tb, valid, row);
            } else if constexpr (MODE == GM_FFN12) {
                if (ti.phase == 0) {
                    epi_swiglu<BN>(p, ti, tb, valid, row);
                    // release this warp's h rows of the tile to the GEMM-2 producers,
                    // which read them with TMA: each lane orders its stores before
                    // later async-proxy accesses, then one release increment
                    __threadfence();
                    fence_proxy_async_global();
                    __syncwarp();
                    if (lane == 0) red_release_gpu_add(p.ready + ti.rt, 1);
                } else {
                    float w = 1.0f;
                    if (valid && p.row_w && row < p.w_rows) w = p.row_w[row];
                    epi_bf16_scaled<BN>(static_cast<uint16_t *>(p.out3), p.N, ti, tb, valid, row, w);
                }
            } else if constexpr (MODE == GM_FFN2 || MODE == GM_DGRAD1) {
                float w = 1.0f;
                if constexpr (MODE == GM_FFN2) {
                    if (valid && p.row_w && row < p.w_rows) w = p.row_w[row];
                }
                epi_bf16_scaled<BN>(static_cast<uint16_t *>(p.out), p.N, ti, tb, valid, row, w);
            } else if constexpr (MODE == GM_DGRAD2) {
                uint16_t *dgu = static_cast<uint16_t *>(p.out2);
                uint16_t *hw = static_cast<uint16_t *>(p.out3);
                float w = 1.0f;
                if (valid && p.row_w && row < p.w_rows) w = p.row_w[row];
                const float cl = p.clamp;
                float dw = 0.0f;
                constexpr int CW2 = BN / (MT::NEPI / 4);   // this warp's columns
                const int c_lo2 = (ew >> 2) * CW2;
                // warps whose 32 rows all exist use TMA stores; a ragged warp must not
                // write past its group (the next rows belong to another tile)
                const bool warp_full = q * 32 + 32 <= ti.rows_valid;
                uint8_t *stg2 = sEpi + (size_t)ew * kEpiWarpBytesDgrad2;
#pragma unroll 1
                for (int c = c_lo2; c < c_lo2 + CW2; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c, r);
                    tmem_wait_ld();
                    uint32_t og[16], ou[16], oh[16];
                    if (valid) {
                        const int col = ti.nt * BN + c;
                        uint16_t *dgd = dgu + (size_t)row * 2 * p.I + col;
                        uint16_t *dud = dgd + p.I;
                        uint16_t *hwd = hw + (size_t)row * p.I + col;
                        // all 16 vector loads of the chunk first: one memory latency per chunk
                        float4 gv4[8], uv4[8];
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            gv4[q4] = *reinterpret_cast<const float4 *>(
                                p.gu_in + gu_offset(row, col + 4 * q4, p.I));
                            uv4[q4] = *reinterpret_cast<const float4 *>(
                                p.gu_in + gu_offset(row, p.I + col + 4 * q4, p.I));
                        }
                        const float *gv = reinterpret_cast<const float *>(gv4);
                        const float *uv = reinterpret_cast<const float *>(uv4);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float dg2[2], du2[2], hw2[2];
#pragma unroll
                            for (int hlf = 0; hlf < 2; ++hlf) {
                                const float g = gv[2 * e + hlf];
                                const float u = uv[2 * e + hlf];
                                const float dA = __uint_as_float(r[2 * e + hlf]);
                                const float a = fminf(g, cl);
                                const float b = fminf(fmaxf(u, -cl), cl);
                                const float sg = sigmoid_fast(a);
                                const float si = a * sg;
                                // bit-identical to the forward's h (same fp32 g, u and code)
                                const float hv = round_bf16(swiglu_clamped(g, u, cl));
                                dw = fmaf(hv, dA, dw);
                                const float dH = w * dA;
                                dg2[hlf] = g <= cl ? dH * b * (sg + a * sg * (1.0f - sg)) : 0.0f;
                                du2[hlf] = (u >= -cl && u <= cl) ? dH * si : 0.0f;
                                hw2[hlf] = w * hv;
                            }
                            og[e] = pack_bf16x2(dg2[0], dg2[1]);
                            ou[e] = pack_bf16x2(du2[0], du2[1]);
                            oh[e] = pack_bf16x2(hw2[0], hw2[1]);
                        }
                        if (!warp_full) {
#pragma unroll
                            for (int q4 = 0; q4 < 16; q4 += 4) {
                                st_global_v4(dgd + 2 * q4, og[q4], og[q4 + 1], og[q4 + 2], og[q4 + 3]);
                                st_global_v4(dud + 2 * q4, ou[q4], ou[q4 + 1], ou[q4 + 2], ou[q4 + 3]);
                                st_global_v4(hwd + 2 * q4, oh[q4], oh[q4 + 1], oh[q4 + 2], oh[q4 + 3]);
                            }
                        }
                    }
                    if (warp_full) {
                        // all 32 rows of this warp exist: stage the three 32 x 32 bf16
                        // blocks (64-byte swizzle) one after the other in the
                        // warp's buffer and write each with a TMA store
                        const uint32_t b0 = smem_u32(stg2);
                        const uint32_t rowb = (uint32_t)lane * 64u;
                        const uint32_t sw2 = (uint32_t)((lane >> 1) & 3);
                        const int col = ti.nt * BN + c;
                        const int wrow = ti.row0 + q * 32;
#pragma unroll
                        for (int which = 0; which < 3; ++which) {
                            const uint32_t *src = which == 0 ? og : (which == 1 ? ou : oh);
                            if (lane == 0) bulk_wait_group_read<0>();
                            __syncwarp();
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                st_shared_v4(b0 + rowb + ((((uint32_t)j) ^ sw2) << 4), src[4 * j],
                                             src[4 * j + 1], src[4 * j + 2], src[4 * j + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                if (which == 0) tma_store_2d(&p.tmO, stg2, col, wrow);
                                else if (which == 1) tma_store_2d(&p.tmO, stg2, p.I + col, wrow);
                                else tma_store_2d(&p.tmO2, stg2, col, wrow);
                                bulk_commit_group();
                            }
                        }
                    }
                }
                // one partial of <h, dA> per (row, column tile, warp half)
                if (valid)
                    p.out4[((size_t)row * p.n_tiles + ti.nt) * (MT::NEPI / 4) + (ew >> 2)] = dw;
            } else {  // GM_WGRAD: fp32 rows through shared memory to coalesced stores
                uint8_t *stg = sEpi + (size_t)ew * kEpiWarpBytes;
                const uint32_t sw = (uint32_t)(lane & 7);
                const bool has_k = ti.kb > 0;
                // this warp's share of the columns
                constexpr int CW = BN / (MT::NEPI / 4);
                const int c_lo = (ew >> 2) * CW;
                // rows [m0 + 32 q, m0 + 32 q + 32) of the group's output, from
                // column nt BN
                const uint64_t pol_out = policy_evict_first();
                float *obase = static_cast<float *>(p.out) +
                               ((size_t)ti.g * p.M + ti.m0 + q * 32) * (size_t)p.N +
                               (size_t)ti.nt * BN;
                auto store_block = [&](const uint32_t (&v)[32], int c) {
                    // transpose through the warp's 4 KB: rows written one per
                    // lane (128-byte swizzle), read back four rows per
                    // instruction, each row leaving as one full 128-byte line
                    const uint32_t sb = smem_u32(stg);
                    __syncwarp();   // every lane has read the previous block back
                    const uint32_t wa = sb + (uint32_t)lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(wa + ((((uint32_t)j) ^ sw) << 4), v[4 * j], v[4 * j + 1],
                                     v[4 * j + 2], v[4 * j + 3]);
                    __syncwarp();
                    const int ch = lane & 7;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = 4 * i + (lane >> 3);
                        const uint4 x = ld_shared_v4(sb + (uint32_t)r * 128u +
                                                     ((uint32_t)(ch ^ (r & 7)) << 4));
                        if constexpr (kWgradL2Hints & 2)
                            st_global_v4_hint(obase + (size_t)r * p.N + c + 4 * ch, x.x, x.y, x.z,
                                              x.w, pol_out);
                        else
                            st_global_v4(obase + (size_t)r * p.N + c + 4 * ch, x.x, x.y, x.z, x.w);
                    }
                };
                // two register sets: the TMEM load of the next block is in flight
                // while the current one is staged
                uint32_t ra[32], rb[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    ra[j] = 0u;
                    rb[j] = 0u;
                }
                if (has_k) {
                    tmem_ld32(tb + c_lo, ra);
                    tmem_wait_ld();
                }
#pragma unroll 1
                for (int c = c_lo; c < c_lo + CW; c += 64) {
                    const bool more1 = c + 32 < c_lo + CW;
                    if (has_k && more1) tmem_ld32(tb + c + 32, rb);
                    store_block(ra, c);
                    if (!more1) break;
                    if (has_k) tmem_wait_ld();
                    if (has_k && c + 64 < c_lo + CW) tmem_ld32(tb + c + 64, ra);
                    store_block(rb, c + 32);
                    if (has_k) tmem_wait_ld();
                }
            }
            tc_fence_before();
            if constexpr (CL == 2) {
                // one arrival per warp on the even CTA's accumulator barrier
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(&tempty[acc]);
                    else mbar_arrive_remote_relaxed(dsmem_map(&tempty[acc], 0));
                }
            } else {
                mbar_arrive(&tempty[acc]);
            }
        }
    }

    if constexpr (TS::TMA_STORE) {
        // the stores must have left shared memory (and landed) before exit
        if (warp >= 2 && lane == 0) bulk_wait_group_all();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (CL == 2) {
        // both CTAs are past their last TMEM read and the pair's MMAs have
        // completed; neither leaves while the other may still signal it
        cluster_sync_all();
        if (warp == 1) tmem_dealloc_pair(tmem_base, TS::TMEM_COLS);
        cluster_sync_all();
    } else {
        if (warp == 1) tmem_dealloc(tmem_base, TS::TMEM_COLS);
    }
}

}  // namespace moe

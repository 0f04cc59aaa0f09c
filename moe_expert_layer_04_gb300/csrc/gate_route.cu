// gate_route.cu -- gate projection, routing and per-modality expert load in
// one kernel ("HyperParallel加速DeepSeek-V4.1多模态1M长序列训练" §2.3, MegaGate:
// score, bias ranking, top-k, score extraction, normalisation and scaling,
// with separate text and vision routing bias; §01 item 5, native multimodal
// MoE: the load of text and vision tokens is balanced separately, so the
// kernel counts the slots each expert receives from either modality).
//
// Work split.  A tile is 128 tokens.  With CS = 2 a cluster of two CTAs takes
// a tile and splits the experts: CTA r accumulates the logits of experts
// [r E/2, (r+1) E/2) in TMEM (tcgen05.mma, M = 128, N = E/2); each CTA loads
// the whole x tile itself (the pair's two reads of it meet in L2).
// With CS = 1 (E not a multiple of 64) one CTA takes all E columns.  TMEM
// holds two accumulators when a CTA's columns fit in 256, so the epilogue of
// one tile overlaps the MMAs of the next.
//
// Epilogue, one token per thread (its TMEM lane), per tile:
//   pass A  each of the CTA's logits (+ offset) goes out through a swizzled
//           staging buffer and a TMA store; its approximate key (fast
//           sigmoid + bias) goes back into the logit's TMEM column.  The
//           maxima of the keys' groups of 4 columns run through a keys-only
//           list of the L largest: its last entry is a lower bound of the
//           L-th largest key (L distinct keys reach it).
//   pass B  the keys come back from TMEM; per 32-expert chunk each lane
//           marks, in a bit mask, the keys above both that bound and the
//           smallest entry of its sorted register list of the L largest
//           (key, id) so far, and inserts only those, so a warp pays for
//           its busiest lane (about 8 candidates of 192 per token instead of
//           35 with one pass).  TMEM is handed back to the MMA warp right
//           after.
//   merge   (CS = 2) rank r owns tokens 64r .. 64r+63 of the tile.  For the
//           other 64 it sends its list to the peer's shared memory
//           (distributed shared memory, bounded mbarrier handshakes); for
//           its own it merges the peer's list into its own.
//   exact   the owner gives the list entries within twice the approximate
//           error of the k-th key the exact key (their logits read back from
//           global memory; sigmoid in fp64 rounded once to fp32, one fp32 add
//           of the bias) and takes the exact top-k among
//           them, equal keys to the lower id.  When the window could reach
//           past the list (many near-equal keys), it rescans the token's
//           logits row from global memory instead (every writer completed and
//           fenced its TMA stores before it signalled).
// This makes the same selection, bit for bit, as the warp-per-token routing
// kernel.  Weights w_j = scaling s_j / sum_i s_i in fp64, rounded once.
// Slot counts per (modality, expert) are summed per CTA in shared memory and
// added to the global counters once per CTA (integer atomics: the result does
// not depend on their order).
#include <cfloat>
#include <climits>
#include <cstring>

#include "moe_ptx.cuh"

namespace moe {
namespace {

constexpr int kGrThreads = 192;      // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kGrKmax = 8;           // largest supported k
constexpr int kGrMaxStages = 4;
constexpr int kGrABytes = 128 * 64 * 2;
constexpr size_t kGrSmemLimit = 227 * 1024;

struct GateRouteParams {
    CUtensorMap tmX;  // x [T, d] bf16, boxes 64 x 128
    CUtensorMap tmW;  // W_g [E, d] bf16, boxes 64 x (columns of one MMA)
    CUtensorMap tmZ;  // logits [T, E] fp32, boxes 32 x 32 (stores)
    const float *offset;  // [E] or null
    const float *bias;    // [2, E] (top-k mode)
    const uint8_t *is_vision;
    const int32_t *input_ids;  // hash mode
    const int32_t *tid2eid;
    const float *logits;  // the output again, for the rare rescan
    int vocab;
    int T, d, E, k, mode, stages;
    float scaling;
    int32_t *ids;
    float *weights, *ssel;
    int32_t *counts;  // [2, E] or null
    int *status;
    long long wait_limit;
};

// Dynamic shared memory: operand stages, 4 x 4 KB logits staging, 4 x 4 KB
// approximate-key staging (one 32 x 32 block per epilogue warp each), 256 B of
// barriers, the merge buffer (2 quadrants x 3 fields x L x 32 floats), then
// offset [E], text bias [E], 4 floats of padding (the two bias rows fall in
// different banks), vision bias [E], counts [2, E].
size_t gr_smem_bytes(int E, int CS, int L, int stages) {
    const size_t stage = kGrABytes + (size_t)(E / CS) * 128;
    return 1024 + (size_t)stages * stage + 8 * 4096 + 256 + (size_t)2 * 3 * L * 32 * 4 +
           (size_t)(3 * E + 4) * 4 + (size_t)2 * E * 4;
}

int gr_stages(int E, int CS, int L) {
    for (int s = kGrMaxStages; s >= 2; --s)
        if (gr_smem_bytes(E, CS, L, s) <= kGrSmemLimit) return s;
    return 0;
}

__device__ __forceinline__ float sigmoid_exact_f(float z) {
    return (float)(1.0 / (1.0 + exp(-(double)z)));
}

// Approximate key from the fast exponential and division: their documented
// error bounds (2 + 1.2|z| ulp for the exponential, 2 ulp for the division)
// put the score within ~3e-7 of the exact one for every z, since the
// exponential's error enters scaled by s(1 - s); the window below allows 4e-6.
__device__ __forceinline__ float approx_key(float z, float b) {
    const float s = __fdividef(1.0f, 1.0f + __expf(-z));
    const float kk = s + b;
    return (kk == kk) ? kk : -FLT_MAX;  // NaN ranks last
}

__device__ __forceinline__ float exact_key(float se, float b) {
    const float kk = __fadd_rn(se, b);
    return (kk == kk) ? kk : -FLT_MAX;
}

// Inserts (key, id) into the descending list when it beats the smallest
// entry, without branches: the new entry sinks from the top and swaps with
// every entry it beats, so it lands after all entries not below it (equal
// keys keep the earlier entry first) and the smallest drops out.
template <int L>
__device__ __forceinline__ void list_insert(float (&kv)[L], int (&iv)[L], float key, int id) {
#pragma unroll
    for (int q = 0; q < L; ++q) {
        const bool sw = key > kv[q];
        const float tk = kv[q];
        const int ti = iv[q];
        kv[q] = sw ? key : tk;
        iv[q] = sw ? id : ti;
        key = sw ? tk : key;
        id = sw ? ti : id;
    }
}

// L: approximate candidates kept per token (more than k); CS: CTAs per tile.
template <int L, int CS>
__global__ void __launch_bounds__(kGrThreads, 1)
    gate_route_kernel(const __grid_constant__ GateRouteParams p) {
    const int E = p.E;
    const int NE = E / CS;                   // columns of this CTA
    const int nmma = NE > 256 ? 2 : 1;
    const int NM = NE / nmma;                // N of one MMA
    const int nacc = NE <= 256 ? 2 : 1;      // accumulators of 256 columns
    const int STAGES = p.stages;
    const int STAGE = kGrABytes + NE * 128;
    const uint32_t idesc = idesc_bf16_f32(128, NM, false, false);
    const int rank = CS == 2 ? (int)cluster_ctarank() : 0;
    const int col0 = rank * NE;
    const int cid = blockIdx.x / CS, ncl = gridDim.x / CS;

    extern __shared__ uint8_t smem_raw[];
    // aligned to 1024 B by pointer arithmetic on the shared array itself, so
    // that the compiler keeps every access derived from it in the shared
    // state space (LDS/STS, shared atomics) instead of generic addressing
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *stages = smem;
    uint8_t *stg_all = smem + (size_t)STAGES * STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(stg_all + 8 * 4096);
    uint64_t *empty = full + kGrMaxStages;
    uint64_t *tfull = empty + kGrMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *lfull = tempty + 2;            // [2]: the peer's list for an owned quadrant
    uint64_t *lempty = lfull + 2;            // [2]: the peer has read our list
    uint64_t *done = lempty + 2;
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_s = reinterpret_cast<volatile int *>(tmem_base_s + 1);
    float *mrg = reinterpret_cast<float *>(stg_all + 8 * 4096 + 256);
    float *s_off = mrg + 2 * 3 * L * 32;
    float *s_bias = s_off + E;   // text row at [0, E), vision row at [E + 4, 2E + 4)
    int *cnt = reinterpret_cast<int *>(s_bias + 2 * E + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);    // released by this CTA's MMAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
            mbar_init(&lfull[a], 32);
            mbar_init(&lempty[a], 32);
        }
        mbar_init(done, 1);
        *abort_s = 0;
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        s_off[i] = p.offset ? p.offset[i] : 0.0f;
        if (p.mode == MOE_ROUTE_TOPK) {
            s_bias[i] = p.bias[i];
            s_bias[E + 4 + i] = p.bias[E + i];
        }
    }
    for (int i = threadIdx.x; i < 2 * E; i += blockDim.x) cnt[i] = 0;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmX);
        tma_prefetch_desc(&p.tmW);
        tma_prefetch_desc(&p.tmZ);
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_s, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the peer's list arrivals target our barriers: both CTAs must have
    // initialised them first
    if constexpr (CS == 2) cluster_sync_all();
    const uint32_t tmem_base = *tmem_base_s;
    const WaitCtl wc{abort_s, p.status, p.wait_limit};
    const int tiles = (p.T + 127) / 128;
    const int kblocks = p.d / 64;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_par[kGrMaxStages];
#pragma unroll
            for (int s = 0; s < kGrMaxStages; ++s) last_par[s] = -1;
            uint32_t s = 0, ph = 0;
            bool ok = true;
            for (int t = cid; ok && t < tiles; t += ncl) {
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], STAGE);
                    uint8_t *a = stages + (size_t)s * STAGE;
                    uint8_t *b = a + kGrABytes;
                    tma_load_2d(a, &p.tmX, &full[s], kb * 64, t * 128);
                    for (int h = 0; h < nmma; ++h)
                        tma_load_2d(b + h * NM * 128, &p.tmW, &full[s], kb * 64, col0 + h * NM);
                    last_par[s] = (int)ph;
                    if (++s == (uint32_t)STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                for (int i = 0; i < STAGES; ++i)
                    if (last_par[i] >= 0)
                        mbar_wait_teardown(&full[i], (uint32_t)last_par[i], p.wait_limit);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        uint32_t s = 0, ph = 0;
        int it = 0;
        bool ok = true;
        for (int t = cid; ok && t < tiles; t += ncl, ++it) {
            const int acc = it % nacc;
            const uint32_t aph = (uint32_t)(it / nacc) & 1u;
            if (!mbar_wait(&tempty[acc], aph ^ 1u, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)acc * 256u;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_addr = smem_u32(stages + (size_t)s * STAGE);
                    const uint32_t b_addr = a_addr + kGrABytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(a_addr + kk * 32, 16, 1024);
                        for (int h = 0; h < nmma; ++h) {
                            const uint64_t bd =
                                sdesc_sw128(b_addr + h * NM * 128 + kk * 32, 16, 1024);
                            umma_bf16(d_tmem + h * NM, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(&empty[s]);
                }
                __syncwarp();
                if (++s == (uint32_t)STAGES) { s = 0; ph ^= 1u; }
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
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int qq = q & 1;             // its slot in the merge buffers
        const bool owner = CS == 1 || (q >> 1) == rank;
        const int k = p.k;
        const bool topk = p.mode == MOE_ROUTE_TOPK;
        uint8_t *stg = stg_all + (size_t)(warp - 2) * 4096;
        const uint32_t stg_row = smem_u32(stg) + (uint32_t)lane * 128u;
        // this lane's row of approximate keys, laid out like its logits row
        uint8_t *krow = stg_all + 4 * 4096 + (size_t)(warp - 2) * 4096 + lane * 128;
        const uint32_t sw = (uint32_t)(lane & 7);
        float *my_mrg = mrg + qq * 3 * L * 32;   // entry i, field f at [(f * L + i) * 32 + lane]
        int it = 0;
        for (int t = cid; t < tiles; t += ncl, ++it) {
            const int acc = it % nacc;
            const uint32_t aph = (uint32_t)(it / nacc) & 1u;
            if (!mbar_wait(&tfull[acc], aph, wc)) break;
            tc_fence_after();
            const int row = t * 128 + q * 32 + lane;
            const bool valid = row < p.T;
            const bool warp_rows = t * 128 + q * 32 < p.T;  // any row of this warp in range
            const int vis = (valid && p.is_vision && p.is_vision[row]) ? 1 : 0;
            const float *bt = s_bias + vis * (E + 4);
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * 256u;

            // hash mode: the table gives the experts up front; each CTA picks
            // the logits of those in its own columns
            int hid[kGrKmax];
            float hz[kGrKmax];
#pragma unroll
            for (int j = 0; j < kGrKmax; ++j) {
                hid[j] = 0;
                hz[j] = 0.0f;
            }
            if (!topk && valid) {
                int tok = p.input_ids[row];
                if (tok < 0 || tok >= p.vocab) {
                    if (owner) record_status(p.status, MOE_ERR_INVALID_ARG);
                    tok = 0;
                }
#pragma unroll
                for (int j = 0; j < kGrKmax; ++j) {
                    if (j < k) {
                        int e = p.tid2eid[(size_t)tok * k + j];
                        if (e < 0 || e >= E) {
                            if (owner) record_status(p.status, MOE_ERR_INVALID_ARG);
                            e = 0;
                        }
                        hid[j] = e;
                    }
                }
            }

            // ---- pass A: logits out; approximate keys back into TMEM; the L
            // largest group-of-4 maxima of the keys
            float gl[L];
#pragma unroll
            for (int j = 0; j < L; ++j) gl[j] = -INFINITY;
            uint32_t ra[32], rb[32];
            tmem_ld32(tb, ra);
            tmem_wait_ld();
#pragma unroll 1
            for (int cc = 0; cc < NE; cc += 32) {
                const int c = col0 + cc;   // expert id of this chunk's first column
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 o = *reinterpret_cast<const float4 *>(s_off + c + j);
                    ra[j] = __float_as_uint(__uint_as_float(ra[j]) + o.x);
                    ra[j + 1] = __float_as_uint(__uint_as_float(ra[j + 1]) + o.y);
                    ra[j + 2] = __float_as_uint(__uint_as_float(ra[j + 2]) + o.z);
                    ra[j + 3] = __float_as_uint(__uint_as_float(ra[j + 3]) + o.w);
                }
                if (warp_rows) {
                    // the previous chunk's store must have read the staging buffer
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stg_row + ((((uint32_t)j) ^ sw) << 4), ra[4 * j],
                                     ra[4 * j + 1], ra[4 * j + 2], ra[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        // rows past T lie outside the tensor and are not written
                        tma_store_2d(&p.tmZ, stg, c, t * 128 + q * 32);
                        bulk_commit_group();
                    }
                }
                if (cc + 32 < NE) tmem_ld32(tb + cc + 32, rb);
                if (topk) {
                    uint32_t kc[32];
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 b4 = *reinterpret_cast<const float4 *>(bt + c + j);
                        kc[j] = __float_as_uint(approx_key(__uint_as_float(ra[j]), b4.x));
                        kc[j + 1] = __float_as_uint(approx_key(__uint_as_float(ra[j + 1]), b4.y));
                        kc[j + 2] = __float_as_uint(approx_key(__uint_as_float(ra[j + 2]), b4.z));
                        kc[j + 3] = __float_as_uint(approx_key(__uint_as_float(ra[j + 3]), b4.w));
                    }
                    tmem_st32(tb + cc, kc);
                    // the L largest group maxima are L distinct keys, so the
                    // L-th largest of them bounds the L-th largest key from below
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        float x = fmaxf(fmaxf(__uint_as_float(kc[4 * g]), __uint_as_float(kc[4 * g + 1])),
                                        fmaxf(__uint_as_float(kc[4 * g + 2]), __uint_as_float(kc[4 * g + 3])));
#pragma unroll
                        for (int i = 0; i < L; ++i) {
                            const float hi = fmaxf(gl[i], x);
                            x = fminf(gl[i], x);
                            gl[i] = hi;
                        }
                    }
                } else if (valid) {
#pragma unroll
                    for (int j = 0; j < kGrKmax; ++j) {
                        const int e = hid[j] - c;
                        if (j < k && e >= 0 && e < 32) {
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj)
                                if (jj == e) hz[j] = __uint_as_float(ra[jj]);
                        }
                    }
                }
                if (cc + 32 < NE) {
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ra[j] = rb[j];
                }
            }

            // ---- pass B (top-k): the keys not below that bound, into the
            // sorted list of the L largest (ids in increasing order)
            float kv[L];
            int iv[L];
#pragma unroll
            for (int j = 0; j < L; ++j) {
                kv[j] = -INFINITY;
                iv[j] = INT_MAX;
            }
            if (topk) {
                tmem_wait_st();
                const float thrg = gl[L - 1];
                tmem_ld32(tb, ra);
                tmem_wait_ld();
#pragma unroll 1
                for (int cc = 0; cc < NE; cc += 32) {
                    const int c = col0 + cc;
                    if (cc + 32 < NE) tmem_ld32(tb + cc + 32, rb);
                    // this lane's keys, for the candidates' reads by index
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4 *>(krow + ((((uint32_t)j) ^ sw) << 4)) =
                            make_uint4(ra[4 * j], ra[4 * j + 1], ra[4 * j + 2], ra[4 * j + 3]);
                    const float thr0 = kv[L - 1];
                    uint32_t m = 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float kk = __uint_as_float(ra[j]);
                        m |= (kk > thr0 && kk >= thrg ? 1u : 0u) << j;
                    }
                    if (!valid) m = 0;
                    // a converged loop: every lane runs the warp's largest count,
                    // lanes out of candidates insert nothing (a divergent loop
                    // costs several times more per trip here)
                    const int trips = __reduce_max_sync(0xffffffffu, __popc(m));
                    for (int r = 0; r < trips; ++r) {
                        const bool act = m != 0u;
                        const int j = act ? __ffs(m) - 1 : 0;
                        m &= m - 1u;
                        const uint32_t off = ((((uint32_t)(j >> 2)) ^ sw) << 4) + (j & 3) * 4;
                        const float key = *reinterpret_cast<const float *>(krow + off);
                        list_insert<L>(kv, iv, act ? key : -INFINITY, c + j);
                    }
                    if (cc + 32 < NE) {
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) ra[j] = rb[j];
                    }
                }
            }
            // TMEM is free for the next tile
            tc_fence_before();
            mbar_arrive(&tempty[acc]);

            // ---- merge the two halves of the experts (CS = 2)
            if constexpr (CS == 2) {
                if (!owner) {
                    // send our list (top-k) or our picked logits (hash) for these 32
                    // tokens, once our logits stores are complete and visible
                    if (!mbar_wait_cluster(&lempty[qq], (uint32_t)(it & 1) ^ 1u, wc)) break;
                    if (lane == 0) {
                        bulk_wait_group_all();
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                    const uint32_t dst = dsmem_map(my_mrg, (uint32_t)(rank ^ 1));
#pragma unroll
                    for (int i = 0; i < L; ++i) {
                        // top-k: the list; hash: the picked logits (field 2)
                        dsmem_st_u32(dst + (uint32_t)((0 * L + i) * 32 + lane) * 4u,
                                     __float_as_uint(kv[i]));
                        dsmem_st_u32(dst + (uint32_t)((1 * L + i) * 32 + lane) * 4u,
                                     (uint32_t)iv[i]);
                        if (!topk)
                            dsmem_st_u32(dst + (uint32_t)((2 * L + i) * 32 + lane) * 4u,
                                         __float_as_uint(i < kGrKmax ? hz[i % kGrKmax] : 0.0f));
                    }
                    mbar_arrive_remote(dsmem_map(&lfull[qq], (uint32_t)(rank ^ 1)));
                    continue;
                }
                // receive the peer's half for our tokens, then free its slot
                if (!mbar_wait_cluster(&lfull[qq], (uint32_t)(it & 1), wc)) break;
                float pk[L], pz[L];
                int pi[L];
#pragma unroll
                for (int i = 0; i < L; ++i) {
                    pk[i] = my_mrg[(0 * L + i) * 32 + lane];
                    pi[i] = __float_as_int(my_mrg[(1 * L + i) * 32 + lane]);
                    pz[i] = topk ? 0.0f : my_mrg[(2 * L + i) * 32 + lane];
                }
                mbar_arrive_remote(dsmem_map(&lempty[qq], (uint32_t)(rank ^ 1)));
                if (topk) {
#pragma unroll
                    for (int i = 0; i < L; ++i) list_insert<L>(kv, iv, pk[i], pi[i]);
                } else {
                    // the peer picked the logits of the experts in its columns
#pragma unroll
                    for (int j = 0; j < kGrKmax; ++j) {
                        const bool theirs = (hid[j] >= NE) != (rank == 1);
                        if (j < k && theirs) hz[j] = pz[j % L];
                    }
                }
            }

            // ---- the exact top-k (owner)
            int my_id[kGrKmax];
            float my_s[kGrKmax];
#pragma unroll
            for (int j = 0; j < kGrKmax; ++j) {
                my_id[j] = 0;
                my_s[j] = 0.0f;
            }
            // the list is sorted: the k-th key is the smallest of the first k
            float kth = kv[0];
#pragma unroll
            for (int j = 1; j < kGrKmax; ++j)
                if (j < k) kth = fminf(kth, kv[j]);
            // error bound of the approximate key: see approx_key; the two key
            // additions add half an ulp of the key each
            const float tol = 4e-6f * fmaxf(1.0f, fabsf(kth));
            const float thr = kth - 2.0f * tol;
            const bool rescan = topk && valid && !(kv[L - 1] < thr);
            if (topk) {
                // the exact keys start from the logits in global memory (the
                // list holds keys and ids only).  Our own stores must be
                // complete and visible first (the peer's are: it fenced them
                // before it signalled).
                if (lane == 0) {
                    bulk_wait_group_all();
                    fence_proxy_async_global();
                }
                __syncwarp();
            }
            if (topk && __any_sync(0xffffffffu, rescan)) {
                // the window may hold experts the list dropped: stream the token's
                // whole logits row through an exact top-k
                if (rescan) {
                    float ek[kGrKmax], es[kGrKmax];
                    int ei[kGrKmax];
#pragma unroll
                    for (int j = 0; j < kGrKmax; ++j) {
                        ek[j] = -INFINITY;
                        es[j] = 0.0f;
                        ei[j] = INT_MAX;
                    }
                    const float *zrow = p.logits + (size_t)row * E;
                    for (int e = 0; e < E; ++e) {
                        const float z = __ldcg(zrow + e);
                        if (!(approx_key(z, bt[e]) >= thr)) continue;
                        const float se = sigmoid_exact_f(z);
                        float key = exact_key(se, bt[e]);
                        // ids arrive in increasing order: an equal key goes after
                        int id = e;
                        float sv = se;
#pragma unroll
                        for (int q2 = 0; q2 < kGrKmax; ++q2) {
                            if (q2 < k && key > ek[q2]) {
                                const float tk = ek[q2];
                                const int ti = ei[q2];
                                const float ts = es[q2];
                                ek[q2] = key;
                                ei[q2] = id;
                                es[q2] = sv;
                                key = tk;
                                id = ti;
                                sv = ts;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < kGrKmax; ++j) {
                        my_id[j] = ei[j] == INT_MAX ? 0 : ei[j];
                        my_s[j] = es[j];
                    }
                }
            }

            if (topk && valid && !rescan) {
                float ek[L], es[L], zw[L];
                const float *zrow = p.logits + (size_t)row * E;
#pragma unroll
                for (int i = 0; i < L; ++i)
                    zw[i] = kv[i] >= thr && (unsigned)iv[i] < (unsigned)E ? __ldcg(zrow + iv[i])
                                                                        : 0.0f;
#pragma unroll
                for (int i = 0; i < L; ++i) {
                    ek[i] = -INFINITY;
                    es[i] = 0.0f;
                    if (kv[i] >= thr) {
                        es[i] = sigmoid_exact_f(zw[i]);
                        ek[i] = exact_key(es[i], bt[iv[i]]);
                    }
                }
                uint32_t taken = 0;
#pragma unroll
                for (int j = 0; j < kGrKmax; ++j) {
                    if (j < k) {
                        float bk = -INFINITY, bv = 0.0f;
                        int bi = INT_MAX;
                        uint32_t bbit = 0;
#pragma unroll
                        for (int i = 0; i < L; ++i) {
                            if (!(taken >> i & 1u) && kv[i] >= thr &&
                                (ek[i] > bk || (ek[i] == bk && iv[i] < bi))) {
                                bk = ek[i];
                                bi = iv[i];
                                bv = es[i];
                                bbit = 1u << i;
                            }
                        }
                        taken |= bbit;
                        my_id[j] = bi == INT_MAX ? 0 : bi;
                        my_s[j] = bv;
                    }
                }
            } else if (!topk && valid) {
#pragma unroll
                for (int j = 0; j < kGrKmax; ++j) {
                    my_id[j] = hid[j];
                    my_s[j] = j < k ? sigmoid_exact_f(hz[j]) : 0.0f;
                }
            }
            if (valid) {
                double S = 0.0;
#pragma unroll
                for (int j = 0; j < kGrKmax; ++j)
                    if (j < k) S += (double)my_s[j];
#pragma unroll
                for (int j = 0; j < kGrKmax; ++j) {
                    if (j < k) {
                        const size_t o = (size_t)row * k + j;
                        p.ids[o] = my_id[j];
                        p.ssel[o] = my_s[j];
                        p.weights[o] =
                            S > 0.0 ? (float)((double)p.scaling * (double)my_s[j] / S) : 0.0f;
                        if (p.counts) atomicAdd(&cnt[vis * E + my_id[j]], 1);
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_group_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (p.counts)
        for (int i = threadIdx.x; i < 2 * E; i += blockDim.x)
            if (cnt[i]) atomicAdd(&p.counts[i], cnt[i]);
    // no CTA of the pair may exit while the other can still write into its
    // shared memory or arrive on its barriers
    if constexpr (CS == 2) cluster_sync_all();
}

template <int L, int CS>
moe_status launch_variant(const GateRouteParams &p, int T, cudaStream_t st) {
    auto kern = gate_route_kernel<L, CS>;
    static bool attr_set[64] = {};
    static int max_clusters[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kGrSmemLimit) != cudaSuccess)
            return MOE_ERR_CUDA;
        if constexpr (CS == 2) {
            // how many CTA pairs can be resident at once
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
            cfg.blockDim = dim3(kGrThreads, 1, 1);
            cfg.dynamicSmemBytes = kGrSmemLimit;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
                return MOE_ERR_CUDA;
            max_clusters[dev] = n;
        }
        attr_set[dev] = true;
    }
    // at least 116 KB: one CTA per SM, so that no CTA waits for another's
    // 512 TMEM columns
    size_t smem = gr_smem_bytes(p.E, CS, L, p.stages);
    if (smem < 116 * 1024) smem = 116 * 1024;
    const int tiles = (T + 127) / 128;
    if constexpr (CS == 1) {
        const int grid = tiles < num_sms() ? tiles : num_sms();
        kern<<<grid, kGrThreads, smem, st>>>(p);
    } else {
        const int clusters = tiles < max_clusters[dev] ? tiles : max_clusters[dev];
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * clusters, 1, 1);
        cfg.blockDim = dim3(kGrThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return cuda_status(cudaGetLastError());
}

// The experts split over a CTA pair when both halves are whole 32-column chunks.
int gr_cluster(int E) { return (E % 64 == 0) ? 2 : 1; }
int gr_list(int k) { return k <= 6 ? 8 : 12; }

}  // namespace

bool gate_route_supported(int T, int d, int E, int k) {
    return T >= 1 && d % 64 == 0 && E % 32 == 0 && E >= 32 && E <= 512 && k >= 1 &&
           k <= kGrKmax && k <= E && gr_stages(E, gr_cluster(E), gr_list(k)) >= 2;
}

moe_status launch_gate_route(const uint16_t *x, const uint16_t *Wg, const float *offset,
                             const float *bias, const uint8_t *is_vision,
                             const int32_t *input_ids, const int32_t *tid2eid, int vocab, int T,
                             int d, int E, int k, float scaling, moe_route_mode mode,
                             float *logits, int32_t *ids, float *weights, float *ssel,
                             int32_t *counts, cudaStream_t st) {
    const int CS = gr_cluster(E), L = gr_list(k);
    GateRouteParams p;
    std::memset(&p, 0, sizeof p);
    const int NE = E / CS;
    const int NM = NE > 256 ? NE / 2 : NE;
    if (!encode_tmap_bf16_2d(&p.tmX, x, d, T, (uint64_t)d * 2, 64, 128))
        return MOE_ERR_CUDA;
    if (!encode_tmap_bf16_2d(&p.tmW, Wg, d, E, (uint64_t)d * 2, 64, NM)) return MOE_ERR_CUDA;
    if (!encode_tmap_f32_2d(&p.tmZ, logits, E, T, (uint64_t)E * 4, 32, 32)) return MOE_ERR_CUDA;
    p.offset = offset;
    p.bias = bias;
    p.is_vision = is_vision;
    p.input_ids = input_ids;
    p.tid2eid = tid2eid;
    p.logits = logits;
    p.vocab = vocab;
    p.T = T;
    p.d = d;
    p.E = E;
    p.k = k;
    p.mode = (int)mode;
    p.stages = gr_stages(E, CS, L);
    p.scaling = scaling;
    p.ids = ids;
    p.weights = weights;
    p.ssel = ssel;
    p.counts = counts;
    p.status = device_status_ptr();
    if (!p.status) return MOE_ERR_CUDA;
    p.wait_limit = kWaitLimitCycles;
    if (counts && cudaMemsetAsync(counts, 0, (size_t)2 * E * sizeof(int32_t), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (CS == 2) return L == 8 ? launch_variant<8, 2>(p, T, st) : launch_variant<12, 2>(p, T, st);
    return L == 8 ? launch_variant<8, 1>(p, T, st) : launch_variant<12, 1>(p, T, st);
}

}  // namespace moe

// combine.cu -- result return and weighted combine, and the token-side steps
// of the backward.
//
//   combine       y[t] = y_perm[S+t] + sum_j y_perm[slot_row[t,j]]
//                 ("HyperParallel加速DeepSeek-V4.1多模态1M长序列训练" §2.3 MegaMoE
//                 "result return"; "Twinkle x 昇腾…" FSDP2-4D: results come back
//                 and are merged by routing weight -- y_perm already carries it)
//   router bwd    dw_j = sum of the dgrad-2 partials of the slot's row;
//                 ds_j = (scaling/S)(dw_j - sum_i dw_i w_i / scaling),
//                 dz_j = ds_j s_j (1 - s_j)   (the normalisation-gradient chain
//                 that MegaGate fuses, same page §2.3)
//   dX assemble   dX[t] = dX_perm[S+t] + sum_j dX_perm[slot_row[t,j]] + sum_j dz_j W_g[ids_j]
//   dW_g          dW_g[e] = sum over the rows of expert e of dz_row * x_perm[row]
//
// All sums are fp32 in a fixed order (gather form, no atomics), so every
// result is deterministic.
#include "moe_ptx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += bf16_lo(w[i]);
        acc[2 * i + 1] += bf16_hi(w[i]);
    }
}

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float a, const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(a, bf16_lo(w[i]), acc[2 * i]);
        acc[2 * i + 1] = fmaf(a, bf16_hi(w[i]), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
    return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                      pack_bf16x2(a[6], a[7]));
}

// One thread per (token, 16-byte column chunk).  KM >= k is a compile-time
// bound: the slot indices and then all k + 1 row loads of the chunk are issued
// before the first add, so a thread waits for one memory latency, not k + 1
// in a row.  The sum is fp32 in a fixed order: shared row first, then the
// slots in order.  KM = 0 is the generic form for any k (one row at a time).
// When dz != nullptr the gate term sum_j dz_j W_g[ids_j] is added as well (the
// dX assembly of the backward), after the slots.  GATE = true (KM > 0) is that
// form: the slot rows, the gate's ids and dz are read together, then all row
// loads (k + 1 rows of dX_perm, k rows of W_g) are issued before the first
// add, so the gate term costs no extra memory latency.
template <int KM, bool GATE = false>
__global__ void __launch_bounds__(256) combine_kernel(const uint4 *__restrict__ yp,
                                                      const int32_t *__restrict__ slot_row,
                                                      int T, int vecs, int k, int with_shared,
                                                      const float *__restrict__ dz,
                                                      const int32_t *__restrict__ ids,
                                                      const uint4 *__restrict__ Wg,
                                                      uint4 *__restrict__ y) {
    const size_t S = (size_t)T * k;
    const size_t n = (size_t)T * vecs;
    for (size_t it = blockIdx.x * (size_t)blockDim.x + threadIdx.x; it < n;
         it += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(it / vecs);
        const int c = (int)(it - (size_t)t * vecs);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        const int32_t *sr = slot_row + (size_t)t * k;
        if constexpr (KM == 0) {
            if (with_shared) add_bf16x8(acc, yp[(S + t) * vecs + c]);
            for (int j = 0; j < k; ++j) add_bf16x8(acc, yp[(size_t)sr[j] * vecs + c]);
            if (dz) {
                for (int j = 0; j < k; ++j)
                    fma_bf16x8(acc, dz[(size_t)t * k + j],
                               Wg[(size_t)ids[(size_t)t * k + j] * vecs + c]);
            }
        } else if constexpr (GATE) {
            int rows[KM], gid[KM];
            float a[KM];
#pragma unroll
            for (int j = 0; j < KM; ++j) {
                rows[j] = j < k ? sr[j] : 0;
                gid[j] = j < k ? ids[(size_t)t * k + j] : 0;
                a[j] = j < k ? dz[(size_t)t * k + j] : 0.0f;
            }
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
            const uint4 vs = with_shared ? yp[(S + t) * vecs + c] : zero;
            uint4 v[KM], w[KM];
#pragma unroll
            for (int j = 0; j < KM; ++j) {
                v[j] = j < k ? yp[(size_t)rows[j] * vecs + c] : zero;
                w[j] = j < k ? Wg[(size_t)gid[j] * vecs + c] : zero;
            }
            if (with_shared) add_bf16x8(acc, vs);
#pragma unroll
            for (int j = 0; j < KM; ++j)
                if (j < k) add_bf16x8(acc, v[j]);
#pragma unroll
            for (int j = 0; j < KM; ++j)
                if (j < k) fma_bf16x8(acc, a[j], w[j]);
        } else {
            int rows[KM];
#pragma unroll
            for (int j = 0; j < KM; ++j) rows[j] = j < k ? sr[j] : 0;
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
            const uint4 vs = with_shared ? yp[(S + t) * vecs + c] : zero;
            uint4 v[KM];
#pragma unroll
            for (int j = 0; j < KM; ++j) v[j] = j < k ? yp[(size_t)rows[j] * vecs + c] : zero;
            if (with_shared) add_bf16x8(acc, vs);
#pragma unroll
            for (int j = 0; j < KM; ++j)
                if (j < k) add_bf16x8(acc, v[j]);
            if (dz) {
                float a[KM];
#pragma unroll
                for (int j = 0; j < KM; ++j) {
                    a[j] = j < k ? dz[(size_t)t * k + j] : 0.0f;
                    rows[j] = j < k ? ids[(size_t)t * k + j] : 0;
                }
#pragma unroll
                for (int j = 0; j < KM; ++j) v[j] = j < k ? Wg[(size_t)rows[j] * vecs + c] : zero;
#pragma unroll
                for (int j = 0; j < KM; ++j)
                    if (j < k) fma_bf16x8(acc, a[j], v[j]);
            }
        }
        y[it] = pack8(acc);
    }
}

// One warp per token, lane j < k owns slot j.
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const float *__restrict__ dw_part, int n_part, const int32_t *__restrict__ slot_row,
    const int32_t *__restrict__ ids, const float *__restrict__ weights,
    const float *__restrict__ ssel, int T, int E, int k, float scaling,
    float *__restrict__ dz_sel, float *__restrict__ dz_row, float *__restrict__ dlogits,
    float *__restrict__ dweights) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nw = gridDim.x * 8;
    for (int t = gw; t < T; t += nw) {
        float dw = 0.0f, s = 0.0f, wt = 0.0f;
        int row = 0, e = 0;
        if (lane < k) {
            const size_t o = (size_t)t * k + lane;
            row = slot_row[o];
            for (int n = 0; n < n_part; ++n) dw += dw_part[(size_t)row * n_part + n];
            s = ssel[o];
            wt = weights[o];
            e = ids[o];
        }
        float Ssum = 0.0f, dot = 0.0f;
        for (int j = 0; j < k; ++j) {
            Ssum += __shfl_sync(0xffffffffu, s, j);
            dot += __shfl_sync(0xffffffffu, dw, j) * __shfl_sync(0xffffffffu, wt, j);
        }
        // w_j = scaling s_j / S  =>  ds_j = (scaling dw_j - sum_i dw_i w_i) / S
        // (no division by the scaling: scaling 0 gives zero gradients)
        float dzv = 0.0f;
        if (Ssum > 0.0f) {
            const float ds = (scaling * dw - dot) / Ssum;
            dzv = ds * s * (1.0f - s);
        }
        if (dlogits) {
            float *dl = dlogits + (size_t)t * E;
            for (int c = lane; c < E; c += 32) dl[c] = 0.0f;
            __syncwarp();
            if (lane < k) dl[e] = dzv;
        }
        if (lane < k) {
            const size_t o = (size_t)t * k + lane;
            dz_sel[o] = dzv;
            dz_row[row] = dzv;
            if (dweights) dweights[o] = dw;
        }
    }
}

// dW_g[e] = sum over expert e's rows of dz_row * x_perm[row].  The rows are
// cut into chunks of kDwgChunk rows that never cross an expert (an expert of
// n rows has ceil(n / kDwgChunk) chunks), so every block streams about the
// same bytes however skewed the load.  Each chunk's sum lands in its own row
// of the workspace; the reduction adds an expert's chunks in chunk order, and
// a chunk sums its rows in row order, so the result does not depend on the
// schedule.
constexpr int kDwgChunk = 256;

// One block of 1024 threads (E <= 1024): chunk_first[e] = chunks before
// expert e (chunk_first[E] = all of them, at most nc_max), chunk_expert[c] =
// the expert of chunk c, -1 for the unused rest of the bound.
__global__ void __launch_bounds__(1024) dwg_plan_kernel(const int32_t *__restrict__ offsets, int E,
                                                        int nc_max, int32_t *__restrict__ chunk_first,
                                                        int32_t *__restrict__ chunk_expert) {
    __shared__ int32_t warp_sum[32];
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    int n = 0;
    if (t < E) {
        const int rows = offsets[t + 1] - offsets[t];
        n = rows > 0 ? (rows + kDwgChunk - 1) / kDwgChunk : 0;
    }
    // inclusive scan of n over the block
    int v = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_sum[wid] = v;
    __syncthreads();
    if (wid == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        warp_sum[lane] = w;
    }
    __syncthreads();
    const int incl = v + (wid > 0 ? warp_sum[wid - 1] : 0);
    const int first = incl - n;
    if (t < E) {
        chunk_first[t] = first < nc_max ? first : nc_max;
        for (int j = 0; j < n && first + j < nc_max; ++j) chunk_expert[first + j] = t;
    }
    if (t == E - 1 || (E == 0 && t == 0)) chunk_first[E] = incl < nc_max ? incl : nc_max;
    const int total = warp_sum[31] < nc_max ? warp_sum[31] : nc_max;
    for (int c = total + t; c < nc_max; c += blockDim.x) chunk_expert[c] = -1;
}

// Block (chunk, 512 columns): 64 threads x 8 columns, eight rows in flight.
__global__ void __launch_bounds__(64) dwg_partial_kernel(const uint4 *__restrict__ xp,
                                                         const float *__restrict__ dz_row,
                                                         const int32_t *__restrict__ offsets,
                                                         const int32_t *__restrict__ chunk_first,
                                                         const int32_t *__restrict__ chunk_expert,
                                                         int vecs, float *__restrict__ part) {
    const int ch = blockIdx.x;
    const int e = chunk_expert[ch];
    const int c = blockIdx.y * 64 + threadIdx.x;
    if (e < 0 || c >= vecs) return;
    const int lo = offsets[e] + (ch - chunk_first[e]) * kDwgChunk;
    const int end = offsets[e + 1];
    const int hi = end < lo + kDwgChunk ? end : lo + kDwgChunk;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int r = lo;
    for (; r + 8 <= hi; r += 8) {
        uint4 v[8];
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = xp[(size_t)(r + j) * vecs + c];
            a[j] = dz_row[r + j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) fma_bf16x8(acc, a[j], v[j]);
    }
    for (; r < hi; ++r) fma_bf16x8(acc, dz_row[r], xp[(size_t)r * vecs + c]);
    float4 *dst = reinterpret_cast<float4 *>(part + ((size_t)ch * vecs + c) * 8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

__device__ __forceinline__ void add4(float4 &a, const float4 b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// One thread per (expert, 4 columns): the expert's chunks in order, four
// loads in flight.  An expert without rows gets zeros.
__global__ void __launch_bounds__(256) dwg_reduce_kernel(const float4 *__restrict__ part,
                                                         const int32_t *__restrict__ chunk_first,
                                                         int E, int d4, float4 *__restrict__ dWg) {
    const size_t n = (size_t)E * d4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const int e = (int)(i / d4);
        const int c = (int)(i - (size_t)e * d4);
        const int f = chunk_first[e], m = chunk_first[e + 1] - f;
        float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        int j = 0;
        for (; j + 4 <= m; j += 4) {
            const float4 b0 = part[(size_t)(f + j) * d4 + c];
            const float4 b1 = part[(size_t)(f + j + 1) * d4 + c];
            const float4 b2 = part[(size_t)(f + j + 2) * d4 + c];
            const float4 b3 = part[(size_t)(f + j + 3) * d4 + c];
            add4(a, b0);
            add4(a, b1);
            add4(a, b2);
            add4(a, b3);
        }
        for (; j < m; ++j) add4(a, part[(size_t)(f + j) * d4 + c]);
        dWg[i] = a;
    }
}

int token_blocks(int T) {
    const int want = (T + 7) / 8;
    const int cap = num_sms() * 8;
    return want < cap ? want : cap;
}

}  // namespace

// Upper bound of the chunks: sum_e ceil(n_e / kDwgChunk) <= S / kDwgChunk + E.
static size_t dwg_chunks_max(int E, long long S) { return (size_t)(S / kDwgChunk) + (size_t)E; }

size_t dwg_workspace_bytes(int d, int E, long long S) {
    const size_t nc = dwg_chunks_max(E, S);
    return (nc * d * 4 + 255) / 256 * 256 + ((size_t)(E + 1) * 4 + 255) / 256 * 256 +
           (nc * 4 + 255) / 256 * 256;
}

moe_status launch_combine(const uint16_t *y_perm, const int32_t *slot_row, int T, int d, int k,
                          int with_shared, const float *dz, const int32_t *ids,
                          const uint16_t *Wg, uint16_t *y, cudaStream_t st) {
    const size_t n = (size_t)T * (d / 8);
    const size_t want = (n + 255) / 256;
    const size_t cap = (size_t)num_sms() * 8;
    const int grid = (int)(want < cap ? want : cap);
    const uint4 *yp = reinterpret_cast<const uint4 *>(y_perm);
    const uint4 *wg = reinterpret_cast<const uint4 *>(Wg);
    uint4 *yo = reinterpret_cast<uint4 *>(y);
    // the gate form holds 2 KM row chunks in registers: KM = 6 (the usual
    // top-6) keeps it at three blocks per SM
    if (k <= 6 && dz)
        combine_kernel<6, true><<<grid, 256, 0, st>>>(yp, slot_row, T, d / 8, k, with_shared, dz,
                                                      ids, wg, yo);
    else if (k <= 8 && dz)
        combine_kernel<8, true><<<grid, 256, 0, st>>>(yp, slot_row, T, d / 8, k, with_shared, dz,
                                                      ids, wg, yo);
    else if (k <= 8)
        combine_kernel<8><<<grid, 256, 0, st>>>(yp, slot_row, T, d / 8, k, with_shared, dz, ids,
                                                wg, yo);
    else
        combine_kernel<0><<<grid, 256, 0, st>>>(yp, slot_row, T, d / 8, k, with_shared, dz, ids,
                                                wg, yo);
    return cuda_status(cudaGetLastError());
}

moe_status launch_router_bwd(const float *dw_part, int n_part, const int32_t *slot_row,
                             const int32_t *ids, const float *weights, const float *ssel, int T,
                             int E, int k, float scaling, float *dz_sel, float *dz_row,
                             float *dlogits, float *dweights, cudaStream_t st) {
    router_bwd_kernel<<<token_blocks(T), 256, 0, st>>>(dw_part, n_part, slot_row, ids, weights,
                                                       ssel, T, E, k, scaling, dz_sel, dz_row,
                                                       dlogits, dweights);
    return cuda_status(cudaGetLastError());
}

moe_status launch_dwg(const uint16_t *x_perm, const float *dz_row, const int32_t *offsets, int d,
                      int E, long long S, float *part, float *dWg, cudaStream_t st) {
    if (E > 1024) return MOE_ERR_UNSUPPORTED;
    const int vecs = d / 8;
    const size_t nc = dwg_chunks_max(E, S);
    if (nc > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    uint8_t *base = reinterpret_cast<uint8_t *>(part);
    int32_t *chunk_first = reinterpret_cast<int32_t *>(base + (nc * d * 4 + 255) / 256 * 256);
    int32_t *chunk_expert =
        reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(chunk_first) +
                                    ((size_t)(E + 1) * 4 + 255) / 256 * 256);
    dwg_plan_kernel<<<1, 1024, 0, st>>>(offsets, E, (int)nc, chunk_first, chunk_expert);
    if (nc > 0) {
        dim3 grid((unsigned)nc, (vecs + 63) / 64);
        dwg_partial_kernel<<<grid, 64, 0, st>>>(reinterpret_cast<const uint4 *>(x_perm), dz_row,
                                                offsets, chunk_first, chunk_expert, vecs, part);
    }
    const int d4 = d / 4;
    const size_t n4 = (size_t)E * d4;
    const int blocks = (int)((n4 + 255) / 256 < (size_t)num_sms() * 8 ? (n4 + 255) / 256
                                                                       : (size_t)num_sms() * 8);
    dwg_reduce_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(part), chunk_first,
                                              E, d4, reinterpret_cast<float4 *>(dWg));
    return cuda_status(cudaGetLastError());
}

}  // namespace moe

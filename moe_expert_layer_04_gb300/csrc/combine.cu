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

// Block (e, column chunk of 512, row split p): partial sums of dz_row * x_perm
// over the split's share of expert e's rows.  64 threads x 8 columns.
__global__ void __launch_bounds__(64) dwg_partial_kernel(const uint4 *__restrict__ xp,
                                                         const float *__restrict__ dz_row,
                                                         const int32_t *__restrict__ offsets,
                                                         int vecs, int E, int splits,
                                                         float *__restrict__ part) {
    const int e = blockIdx.x;
    const int c = blockIdx.y * 64 + threadIdx.x;
    const int sp = blockIdx.z;
    const int lo = offsets[e], hi = offsets[e + 1];
    const int n = hi - lo;
    const int r0 = lo + (int)((long long)n * sp / splits);
    const int r1 = lo + (int)((long long)n * (sp + 1) / splits);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (c < vecs) {
        int r = r0;
        // four rows in flight per step, summed in row order
        for (; r + 4 <= r1; r += 4) {
            const uint4 v0 = xp[(size_t)r * vecs + c];
            const uint4 v1 = xp[(size_t)(r + 1) * vecs + c];
            const uint4 v2 = xp[(size_t)(r + 2) * vecs + c];
            const uint4 v3 = xp[(size_t)(r + 3) * vecs + c];
            fma_bf16x8(acc, dz_row[r], v0);
            fma_bf16x8(acc, dz_row[r + 1], v1);
            fma_bf16x8(acc, dz_row[r + 2], v2);
            fma_bf16x8(acc, dz_row[r + 3], v3);
        }
        for (; r < r1; ++r) fma_bf16x8(acc, dz_row[r], xp[(size_t)r * vecs + c]);
        float4 *dst = reinterpret_cast<float4 *>(part + (((size_t)sp * E + e) * vecs + c) * 8);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

__global__ void __launch_bounds__(256) dwg_reduce_kernel(const float4 *__restrict__ part,
                                                         size_t n4, int splits,
                                                         float4 *__restrict__ dWg) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        float4 a = part[i];
        for (int sp = 1; sp < splits; ++sp) {
            const float4 b = part[(size_t)sp * n4 + i];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        dWg[i] = a;
    }
}

int token_blocks(int T) {
    const int want = (T + 7) / 8;
    const int cap = num_sms() * 8;
    return want < cap ? want : cap;
}

}  // namespace

// Row splits of each expert's dW_g sum: the hottest expert of a skewed load
// holds ~40 % of a 64K-token slice's rows, and each split is one block.
constexpr int kDwgSplits = 32;

size_t dwg_workspace_bytes(int d, int E) {
    return ((size_t)kDwgSplits * E * d * 4 + 255) / 256 * 256;
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
                      int E, float *part, float *dWg, cudaStream_t st) {
    const int vecs = d / 8;
    dim3 grid(E, (vecs + 63) / 64, kDwgSplits);
    dwg_partial_kernel<<<grid, 64, 0, st>>>(reinterpret_cast<const uint4 *>(x_perm), dz_row,
                                            offsets, vecs, E, kDwgSplits, part);
    const size_t n4 = (size_t)E * d / 4;
    const int blocks = (int)((n4 + 255) / 256 < (size_t)num_sms() * 8 ? (n4 + 255) / 256
                                                                       : (size_t)num_sms() * 8);
    dwg_reduce_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(part), n4,
                                              kDwgSplits, reinterpret_cast<float4 *>(dWg));
    return cuda_status(cudaGetLastError());
}

}  // namespace moe

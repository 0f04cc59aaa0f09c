// permute.cu -- token dispatch on one GPU ("HyperParallel加速DeepSeek-V4.1多模态
// 1M长序列训练" §2.3 MegaMoE "token dispatch"; "Twinkle x 昇腾…" FSDP2-4D: the
// selected experts, from top-k or from the hash table, feed one dispatch).
//
// The T*k routed slots are ordered expert-major, then by token, then by slot
// -- a stable order that needs no atomics to be deterministic:
//   hist     one block per chunk of 4096 slots: per-chunk expert histogram
//   scan     per expert, exclusive prefix over chunks; exclusive prefix over
//            experts -> offsets; absolute start of every (chunk, expert)
//   scatter  inside a chunk, warps take 32 slots at a time in order; equal
//            experts inside a warp are ranked with __match_any_sync, and warps
//            advance the per-expert cursors one after the other
//   gather   one warp per token reads the token's row of x once and writes it
//            to its k routed rows and to its shared-expert row S + t, in
//            16-byte vectors
#include "moe_ptx.cuh"

namespace moe {
namespace {

constexpr int kChunk = 4096;
constexpr int kPermThreads = 256;

__global__ void __launch_bounds__(kPermThreads) perm_hist_kernel(const int32_t *__restrict__ ids,
                                                                 int S, int E,
                                                                 int32_t *__restrict__ part,
                                                                 int *status) {
    extern __shared__ int hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int lo = blockIdx.x * kChunk;
    const int hi = min(S, lo + kChunk);
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        const int e = ids[i];
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
        else record_status(status, MOE_ERR_INVALID_ARG);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) part[(size_t)blockIdx.x * E + e] = hist[e];
}

// One block of 1024 threads; thread e owns expert e.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t *__restrict__ part, int nchunks,
                                                         int S, int T, int E,
                                                         int32_t *__restrict__ counts,
                                                         int32_t *__restrict__ offsets) {
    __shared__ int wsum[32];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        // 8 independent loads in flight per step; the running sum follows
        for (int b0 = 0; b0 < nchunks; b0 += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = b0 + u < nchunks ? part[(size_t)(b0 + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (b0 + u < nchunks) part[(size_t)(b0 + u) * E + e] = run;
                run += v[u];
            }
        }
        counts[e] = run;
    }
    // block-wide exclusive scan of run over experts
    const int lane = e & 31, wid = e >> 5;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = wsum[lane];
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        wsum[lane] = inc - v;
    }
    __syncthreads();
    const int excl = wsum[wid] + incl - run;
    if (e < E) {
        offsets[e] = excl;
        for (int b = 0; b < nchunks; ++b) part[(size_t)b * E + e] += excl;
    }
    if (e == 0) {
        offsets[E] = S;
        offsets[E + 1] = S + T;
    }
}

__global__ void __launch_bounds__(kPermThreads) perm_scatter_kernel(
    const int32_t *__restrict__ ids, const float *__restrict__ weights,
    const int32_t *__restrict__ part, int S, int T, int E, int k, int32_t *__restrict__ row_token,
    int32_t *__restrict__ slot_row, float *__restrict__ row_weight) {
    extern __shared__ int cursor[];
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cursor[e] = part[(size_t)blockIdx.x * E + e];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int lo = blockIdx.x * kChunk;
    const int hi = min(S, lo + kChunk);
    for (int base = lo; base < hi; base += kPermThreads) {
        const int i = base + threadIdx.x;
        int e = -1;
        if (i < hi) {
            e = ids[i];
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt);
        const int cnt = __popc(same);
        for (int w = 0; w < kPermThreads / 32; ++w) {
            if (warp == w && e >= 0) {
                const int pos = cursor[e] + rank;
                __syncwarp(same);
                if (rank == 0) cursor[e] += cnt;
                row_token[pos] = i / k;
                slot_row[i] = pos;
                if (row_weight) row_weight[pos] = weights[i];
            }
            __syncthreads();
        }
    }
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x)
        row_token[S + t] = t;
}

// dst[slot_row[t*k + j]] = src[t] for j < k, and dst[S + t] = src[t].
template <int UNROLL>
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4 *__restrict__ src,
                                                          const int32_t *__restrict__ slot_row,
                                                          int T, int vecs, int k, uint4 *dst) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nw = gridDim.x * 8;
    const size_t S = (size_t)T * k;
    for (int t = gw; t < T; t += nw) {
        int row = 0;
        if (lane < k) row = slot_row[(size_t)t * k + lane];
        const uint4 *s = src + (size_t)t * vecs;
        // every lane runs the same iterations: the shuffles below need the full warp
        for (int c0 = 0; c0 < vecs; c0 += 32 * UNROLL) {
            uint4 v[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < vecs) v[u] = s[c];
            }
            for (int j = 0; j <= k; ++j) {
                const size_t r = j < k ? (size_t)__shfl_sync(0xffffffffu, row, j) : S + t;
                uint4 *d = dst + r * vecs;
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    const int c = c0 + lane + 32 * u;
                    if (c < vecs) d[c] = v[u];
                }
            }
        }
    }
}

}  // namespace

size_t permute_workspace_bytes(int T, int E, int k) {
    const size_t S = (size_t)T * k;
    const size_t nchunks = (S + kChunk - 1) / kChunk;
    return (nchunks * (size_t)E * 4 + 255) / 256 * 256;
}

moe_status launch_gather_rows(const uint16_t *src, const int32_t *slot_row, int T, int d, int k,
                              uint16_t *dst, cudaStream_t st) {
    const int vecs = d / 8;
    const int want = (T + 7) / 8;
    const int blocks = want < num_sms() * 8 ? want : num_sms() * 8;
    gather_rows_kernel<4><<<blocks, 256, 0, st>>>(reinterpret_cast<const uint4 *>(src), slot_row,
                                                  T, vecs, k, reinterpret_cast<uint4 *>(dst));
    return cuda_status(cudaGetLastError());
}

moe_status launch_permute(const int32_t *ids, const float *weights, const uint16_t *x, int T,
                          int d, int E, int k, int32_t *counts, int32_t *offsets,
                          int32_t *row_token, int32_t *slot_row, float *row_weight,
                          uint16_t *x_perm, void *ws, cudaStream_t st) {
    const int S = T * k;
    const int nchunks = (S + kChunk - 1) / kChunk;
    int32_t *part = static_cast<int32_t *>(ws);
    int *status = device_status_ptr();
    if (!status) return MOE_ERR_CUDA;
    const size_t hsmem = (size_t)E * sizeof(int);
    perm_hist_kernel<<<nchunks, kPermThreads, hsmem, st>>>(ids, S, E, part, status);
    perm_scan_kernel<<<1, 1024, 0, st>>>(part, nchunks, S, T, E, counts, offsets);
    perm_scatter_kernel<<<nchunks, kPermThreads, hsmem, st>>>(ids, weights, part, S, T, E, k,
                                                              row_token, slot_row, row_weight);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (x_perm) return launch_gather_rows(x, slot_row, T, d, k, x_perm, st);
    return MOE_OK;
}

}  // namespace moe

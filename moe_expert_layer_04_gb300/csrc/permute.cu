// permute.cu -- token dispatch on one GPU ("HyperParallel加速DeepSeek-V4.1多模态
// 1M长序列训练" §2.3 MegaMoE "token dispatch"; "Twinkle x 昇腾…" FSDP2-4D: the
// selected experts, from top-k or from the hash table, feed one dispatch).
//
// The T*k routed slots are ordered expert-major, then by token, then by slot
// -- a stable order that needs no atomics to be deterministic.  Every step is
// parallel over slots:
//   rank     one block per chunk of 256 slots: each slot's rank among the
//            chunk's slots of the same expert (warp match + earlier warps'
//            counts) and the chunk's expert histogram
//   scan     one block per expert: exclusive prefix of its histogram over the
//            chunks, and its total count
//   scatter  one thread per slot: row = offsets[e] + chunk base + rank, with
//            offsets the exclusive prefix of the counts over experts
//   gather   one warp per token reads the token's row of x once and writes it
//            to its k routed rows and to its shared-expert row S + t, in
//            16-byte vectors
#include <mutex>

#include "moe_ptx.cuh"

namespace moe {
namespace {

constexpr int kChunk = 256;   // slots per block of the rank kernel (one per thread)
constexpr int kPermThreads = 256;

// Block c takes slots [256c, 256c + 256), one per thread.  Equal experts
// inside a warp are ranked with __match_any_sync; warps before this one add
// their counts for the same expert.  Writes the slot's rank inside
// (chunk, expert) into slot_row (the scatter adds the bases later) and the
// chunk's expert histogram into part[c][e].
__global__ void __launch_bounds__(kPermThreads) perm_rank_kernel(const int32_t *__restrict__ ids,
                                                                 int S, int E,
                                                                 int32_t *__restrict__ part,
                                                                 int32_t *__restrict__ local_rank,
                                                                 int *status) {
    extern __shared__ int wcnt[];  // [8][E]
    constexpr int NW = kPermThreads / 32;
    for (int i = threadIdx.x; i < NW * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kChunk + threadIdx.x;
    int e = -1;
    if (i < S) {
        e = ids[i];
        if (e < 0 || e >= E) {
            record_status(status, MOE_ERR_INVALID_ARG);
            e = -1;
        }
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
        int r = rank;
        for (int w = 0; w < warp; ++w) r += wcnt[w * E + e];
        local_rank[i] = r;
    }
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) c += wcnt[w * E + x];
        part[(size_t)blockIdx.x * E + x] = c;
    }
}

// Block e: exclusive prefix of part[c][e] over the chunks c, in place, and
// the expert's total count.
__global__ void __launch_bounds__(kPermThreads) perm_chunk_scan_kernel(int32_t *__restrict__ part,
                                                                       int nchunks, int E,
                                                                       int32_t *__restrict__ counts) {
    __shared__ int wsum[kPermThreads / 32];
    const int e = blockIdx.x;
    const int per = (nchunks + kPermThreads - 1) / kPermThreads;
    const int c0 = threadIdx.x * per;
    // up to kHeld counts stay in registers between the two passes, loaded
    // together (one memory latency instead of one per chunk)
    constexpr int kHeld = 8;
    int held[kHeld];
#pragma unroll
    for (int u = 0; u < kHeld; ++u)
        held[u] = u < per && c0 + u < nchunks ? part[(size_t)(c0 + u) * E + e] : 0;
    int local = 0;
#pragma unroll
    for (int u = 0; u < kHeld; ++u) local += held[u];
    for (int c = c0 + kHeld; c < c0 + per && c < nchunks; ++c) local += part[(size_t)c * E + e];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < wid; ++w) before += wsum[w];
    int run = before + incl - local;
#pragma unroll
    for (int u = 0; u < kHeld; ++u) {
        if (u < per && c0 + u < nchunks) {
            part[(size_t)(c0 + u) * E + e] = run;
            run += held[u];
        }
    }
    for (int c = c0 + kHeld; c < c0 + per && c < nchunks; ++c) {
        const int v = part[(size_t)c * E + e];
        part[(size_t)c * E + e] = run;
        run += v;
    }
    if (threadIdx.x == kPermThreads - 1) counts[e] = run;
}

// Exclusive prefix of counts[0..E) into sh[0..E) by one block (E <= 1024).
__device__ void block_offsets(const int32_t *__restrict__ counts, int E, int *sh) {
    __shared__ int wsum[kPermThreads / 32];
    constexpr int PER = 4;  // 256 threads x 4 >= 1024 experts
    const int e0 = threadIdx.x * PER;
    int v[PER], local = 0;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        v[u] = e0 + u < E ? counts[e0 + u] : 0;
        local += v[u];
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < wid; ++w) run += wsum[w];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        if (e0 + u < E) sh[e0 + u] = run;
        run += v[u];
    }
    __syncthreads();
}

// One thread per slot: row = offsets[e] + chunk base + rank in the chunk.
__global__ void __launch_bounds__(kPermThreads) perm_scatter_kernel(
    const int32_t *__restrict__ ids, const float *__restrict__ weights,
    const int32_t *__restrict__ part, const int32_t *__restrict__ counts, int S, int T, int E,
    int k, int32_t *__restrict__ offsets, int32_t *__restrict__ row_token,
    int32_t *__restrict__ slot_row, float *__restrict__ row_weight) {
    extern __shared__ int off[];  // [E]
    block_offsets(counts, E, off);
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = off[e];
        if (threadIdx.x == 0) {
            offsets[E] = S;
            offsets[E + 1] = S + T;
        }
    }
    const int i = blockIdx.x * kChunk + threadIdx.x;
    if (i < S) {
        const int e = ids[i];
        if (e >= 0 && e < E) {
            const int pos = off[e] + part[(size_t)blockIdx.x * E + e] + slot_row[i];
            row_token[pos] = i / k;
            slot_row[i] = pos;
            if (row_weight) row_weight[pos] = weights[i];
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
    // eight 16-byte loads in flight per lane (56 registers): 4 -> 8 took the
    // 64K-token gathers from 90 to 92-94 % of the copy bandwidth
    gather_rows_kernel<8><<<blocks, 256, 0, st>>>(reinterpret_cast<const uint4 *>(src), slot_row,
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
    perm_rank_kernel<<<nchunks, kPermThreads, (size_t)(kPermThreads / 32) * E * sizeof(int), st>>>(
        ids, S, E, part, slot_row, status);
    perm_chunk_scan_kernel<<<E, kPermThreads, 0, st>>>(part, nchunks, E, counts);
    perm_scatter_kernel<<<nchunks, kPermThreads, (size_t)E * sizeof(int), st>>>(
        ids, weights, part, counts, S, T, E, k, offsets, row_token, slot_row, row_weight);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (x_perm) return launch_gather_rows(x, slot_row, T, d, k, x_perm, st);
    return MOE_OK;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free variant of moe_permute.
//
// The only scratch memory moe_permute needs is the per-(chunk, expert)
// histogram that the rank / scan / scatter kernels share.  Here it lives in a
// file-scope device array instead of the caller's workspace, so a caller that
// cannot allocate device memory can still run the dispatch.  Every GPU that
// loads this library keeps the array (kNoAllocScratchInts * 4 bytes = 4 MiB)
// until the process exits.
namespace moe {
namespace {

constexpr size_t kNoAllocScratchInts = (size_t)1 << 20;
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchInts];

std::mutex g_noalloc_mu;
int32_t *g_noalloc_ptr[64];

// Device address of the scratch array on the current device.  Host code only
// sees a host-side stand-in under the array's name, so the real address is
// asked for once per device (with that device current) and cached.
int32_t *noalloc_scratch() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        int32_t *p = nullptr;
        if (cudaGetSymbolAddress((void **)&p, g_noalloc_scratch) != cudaSuccess || !p)
            return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const int32_t *ids, const float *weights,
                                          const uint16_t *x, int T, int d, int E, int k,
                                          int32_t *counts, int32_t *offsets, int32_t *row_token,
                                          int32_t *slot_row, float *row_weight, uint16_t *x_perm,
                                          void *stream) {
    using namespace moe;
    if (T < 1 || E < 1 || k < 1 || k > E || d < 1) return MOE_ERR_INVALID_ARG;
    if (k > 32 || E > 1024 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k + T >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    if (!ids || !counts || !offsets || !row_token || !slot_row) return MOE_ERR_INVALID_ARG;
    if (row_weight && !weights) return MOE_ERR_INVALID_ARG;
    if (x_perm && (!x || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
    // the histogram needs ceil(T*k / 256) * E ints of the fixed array
    if (permute_workspace_bytes(T, E, k) > kNoAllocScratchInts * sizeof(int32_t))
        return MOE_ERR_UNSUPPORTED;
    int32_t *scratch = noalloc_scratch();
    if (!scratch) return MOE_ERR_CUDA;
    // every histogram entry the scatter reads is written earlier in the same
    // call, so nothing in the array has to start at zero
    return launch_permute(ids, weights, x, T, d, E, k, counts, offsets, row_token, slot_row,
                          row_weight, x_perm, scratch, static_cast<cudaStream_t>(stream));
}

// exchange.cu -- row movement for expert parallelism across GPUs
// ("Twinkle x 昇腾，率先实现Deepseek-V4系列模型高效训练", FSDP2-4D: tokens are
// dispatched to the rank that owns their expert, computed there, returned
// with an all-to-all and combined by routing weight; "HyperParallel加速
// DeepSeek-V4.1多模态1M长序列训练" §2.3 MegaMoE: dispatch and return around
// the expert matmuls).
//
// The exchange itself is a collective of the caller's communication library;
// these kernels only reorder rows in this GPU's memory around it:
//   gather rows   dst[i] = src[idx[i]] (rows of any multiple of 4 bytes; a
//                 negative index writes a zero row), used to regroup the rows
//                 received from every source rank by expert, and back
//   row sums      out[r] = sum of the n partial sums of row r
#include "moe_ptx.cuh"

namespace moe {
namespace {

// One warp per output row; 16-byte vectors when the row allows them.
template <typename V>
__global__ void __launch_bounds__(256) index_gather_kernel(const V *__restrict__ src,
                                                           const int32_t *__restrict__ idx,
                                                           long long n, long long n_src, int vecs,
                                                           V *__restrict__ dst, int *status) {
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * 8;
    for (long long i = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); i < n; i += nw) {
        const int j = idx[i];
        V *d = dst + i * vecs;
        if (j >= n_src) {
            if (lane == 0) record_status(status, MOE_ERR_INVALID_ARG);
            continue;   // an out-of-range index leaves its row unwritten
        }
        if (j < 0) {
            for (int c = lane; c < vecs; c += 32) d[c] = V{};
            continue;
        }
        const V *s = src + (long long)j * vecs;
        for (int c = lane; c < vecs; c += 32) d[c] = s[c];
    }
}

__global__ void __launch_bounds__(256) row_sum_kernel(const float *__restrict__ part, long long n,
                                                      int n_part, float *__restrict__ out) {
    for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < n;
         r += (long long)gridDim.x * blockDim.x) {
        float s = 0.0f;
        for (int q = 0; q < n_part; ++q) s += part[r * n_part + q];
        out[r] = s;
    }
}

}  // namespace

moe_status launch_index_gather(const void *src, const int32_t *idx, long long n, long long n_src,
                               int row_bytes, void *dst, cudaStream_t st) {
    if (n == 0) return MOE_OK;
    int *status = device_status_ptr();
    if (!status) return MOE_ERR_CUDA;
    const long long warps_needed = n;
    const int blocks = (int)(warps_needed < 8LL * 4 * num_sms() ? (warps_needed + 7) / 8
                                                                : 4LL * num_sms());
    const bool v16 = row_bytes % 16 == 0 && aligned16(src) && aligned16(dst);
    if (v16) {
        index_gather_kernel<uint4><<<blocks, 256, 0, st>>>(
            static_cast<const uint4 *>(src), idx, n, n_src, row_bytes / 16,
            static_cast<uint4 *>(dst), status);
    } else {
        index_gather_kernel<uint32_t><<<blocks, 256, 0, st>>>(
            static_cast<const uint32_t *>(src), idx, n, n_src, row_bytes / 4,
            static_cast<uint32_t *>(dst), status);
    }
    return cuda_status(cudaGetLastError());
}

moe_status launch_row_sum(const float *part, long long n, int n_part, float *out,
                          cudaStream_t st) {
    if (n == 0) return MOE_OK;
    const long long blocks_needed = (n + 255) / 256;
    const int blocks = (int)(blocks_needed < 4LL * num_sms() ? blocks_needed : 4LL * num_sms());
    row_sum_kernel<<<blocks, 256, 0, st>>>(part, n, n_part, out);
    return cuda_status(cudaGetLastError());
}

}  // namespace moe

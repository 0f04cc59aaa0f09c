// route.cu -- the routing step: gate projection, score, bias ranking, top-k,
// score extraction, normalisation and scaling ("HyperParallel加速DeepSeek-V4.1
// 多模态1M长序列训练" §2.3, MegaGate bullet, with separate text and vision
// routing bias), and the hash router that looks experts up in
// tid2eid[input_ids] but still weights them with the gate logits ("Twinkle x
// 昇腾，率先实现Deepseek-V4系列模型高效训练", FSDP2-4D section).
//
// One warp per token.  The ranking has to agree bit for bit with a reference
// that evaluates the sigmoid in fp64 and rounds once to fp32, but fp64 is slow
// on this GPU, so the warp ranks in two passes:
//   1. every expert: a fp32 score from expf (a few ulp of error), its key, and
//      the k-th largest such key;
//   2. only the experts whose approximate key lies within twice the error
//      bound of that k-th key (almost always just the k winners) get the
//      exact key: the sigmoid in fp64 rounded to fp32, plus the bias in one
//      fp32 add.  The top-k of the exact keys among them is the answer, since
//      every true winner is inside that window.  The window's experts are
//      packed one per lane first: fp64 runs at a small fraction of the fp32
//      rate here, and a warp pays for every fp64 sequence any lane needs.
// Ties go to the lower expert id.  Weights: w_j = scaling * s_j / sum_i s_i
// with the sum and quotient in fp64, rounded to fp32.
#include <cfloat>
#include <climits>

#include "moe_ptx.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

// Warp argmax of (key, id): larger key wins, equal keys go to the lower id.
__device__ __forceinline__ void warp_argmax(float &key, int &id) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float k2 = __shfl_xor_sync(0xffffffffu, key, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, id, o);
        if (k2 > key || (k2 == key && i2 < id)) {
            key = k2;
            id = i2;
        }
    }
}

__device__ __forceinline__ float sigmoid_exact(float z) {
    return (float)(1.0 / (1.0 + exp(-(double)z)));
}

// Fills slot j = lane (< k) of token t from the selected id and its score.
__device__ __forceinline__ void write_weights(int t, int k, int lane, int my_id, float my_s,
                                             float scaling, int32_t *ids, float *w, float *ssel) {
    double S = 0.0;
    for (int j = 0; j < k; ++j) S += (double)__shfl_sync(0xffffffffu, my_s, j);
    if (lane < k) {
        const size_t o = (size_t)t * k + lane;
        ids[o] = my_id;
        ssel[o] = my_s;
        w[o] = S > 0.0 ? (float)((double)scaling * (double)my_s / S) : 0.0f;
    }
}

template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(
    const float *__restrict__ z, const float *__restrict__ bias,
    const uint8_t *__restrict__ is_vision, int T, int E, int k, float scaling,
    int32_t *__restrict__ ids, float *__restrict__ w, float *__restrict__ ssel) {
    __shared__ int s_e[kRouteWarps][32];
    __shared__ float s_z[kRouteWarps][32], s_b[kRouteWarps][32];
    const int lane = threadIdx.x & 31;
    int *lst_e = s_e[threadIdx.x >> 5];
    float *lst_z = s_z[threadIdx.x >> 5];
    float *lst_b = s_b[threadIdx.x >> 5];
    const int gw = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    const int nw = gridDim.x * kRouteWarps;
    for (int t = gw; t < T; t += nw) {
        const float *zt = z + (size_t)t * E;
        const float *bt = bias + ((is_vision && is_vision[t]) ? E : 0);
        float zv[EPL], key[EPL], bv[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                zv[i] = zt[e];
                bv[i] = bt[e];
                const float s = 1.0f / (1.0f + expf(-zv[i]));
                const float kk = s + bv[i];
                key[i] = (kk == kk) ? kk : -FLT_MAX;  // NaN ranks last
            } else {
                zv[i] = 0.0f;
                bv[i] = 0.0f;
                key[i] = -INFINITY;
            }
        }
        // pass 1: approximate k-th key
        uint32_t taken = 0;
        float kth = INFINITY;
        for (int j = 0; j < k; ++j) {
            float bk = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !(taken >> i & 1u) && (key[i] > bk || (key[i] == bk && e < be))) {
                    bk = key[i];
                    be = e;
                }
            }
            warp_argmax(bk, be);
            if (be != INT_MAX && (be & 31) == lane) taken |= 1u << (be >> 5);
            kth = bk;
        }
        // error bound of the approximate key: expf, 1+e and the division add a
        // few ulp of the score; the two key additions half an ulp of the key each
        const float tol = 4e-6f * fmaxf(1.0f, fabsf(kth));
        const float thr = kth - 2.0f * tol;
        // pass 2: exact keys inside the window, then the exact top-k.  The
        // window's experts are first packed one per lane, so that the warp
        // evaluates the fp64 sigmoid once for all of them.
        bool cand[EPL];
        int ncand = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            cand[i] = e < E && key[i] >= thr;
            ncand += __popc(__ballot_sync(0xffffffffu, cand[i]));
        }
        int my_id = 0;
        float my_s = 0.0f;
        if (ncand <= 32) {
            int base = 0;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const unsigned m = __ballot_sync(0xffffffffu, cand[i]);
                if (cand[i]) {
                    const int pos = base + __popc(m & ((1u << lane) - 1u));
                    lst_e[pos] = lane + 32 * i;
                    lst_z[pos] = zv[i];
                    lst_b[pos] = bv[i];
                }
                base += __popc(m);
            }
            __syncwarp();
            int ce = INT_MAX;
            float cs = 0.0f, ck = -INFINITY;
            if (lane < ncand) {
                ce = lst_e[lane];
                cs = sigmoid_exact(lst_z[lane]);
                const float kk = __fadd_rn(cs, lst_b[lane]);
                ck = (kk == kk) ? kk : -FLT_MAX;
            }
            __syncwarp();
            for (int j = 0; j < k; ++j) {
                float bk = ck;
                int be = ce;
                warp_argmax(bk, be);
                const unsigned owner = __ballot_sync(0xffffffffu, ce == be && be != INT_MAX);
                const int ol = owner ? __ffs(owner) - 1 : 0;
                const float sv = __shfl_sync(0xffffffffu, cs, ol);
                if (lane == ol) {
                    ck = -INFINITY;
                    ce = INT_MAX;
                }
                if (lane == j) {
                    my_id = be == INT_MAX ? 0 : be;
                    my_s = sv;
                }
            }
        } else {
            // many exact ties in the window: every lane evaluates its own experts
            float ek[EPL], es[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                es[i] = 0.0f;
                ek[i] = -INFINITY;
                if (cand[i]) {
                    es[i] = sigmoid_exact(zv[i]);
                    const float kk = __fadd_rn(es[i], bv[i]);
                    ek[i] = (kk == kk) ? kk : -FLT_MAX;
                }
            }
            taken = 0;
            for (int j = 0; j < k; ++j) {
                float bk = -INFINITY;
                int be = INT_MAX;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && !(taken >> i & 1u) && (ek[i] > bk || (ek[i] == bk && e < be))) {
                        bk = ek[i];
                        be = e;
                    }
                }
                warp_argmax(bk, be);
                float sv = 0.0f;
                if (be != INT_MAX && (be & 31) == lane) {
                    const int i = be >> 5;
                    taken |= 1u << i;
#pragma unroll
                    for (int ii = 0; ii < EPL; ++ii)
                        if (ii == i) sv = es[ii];
                }
                const int owner = be == INT_MAX ? 0 : (be & 31);
                sv = __shfl_sync(0xffffffffu, sv, owner);
                if (lane == j) {
                    my_id = be == INT_MAX ? 0 : be;
                    my_s = sv;
                }
            }
        }
        write_weights(t, k, lane, my_id, my_s, scaling, ids, w, ssel);
    }
}

__global__ void __launch_bounds__(kRouteWarps * 32) route_hash_kernel(
    const float *__restrict__ z, const int32_t *__restrict__ input_ids,
    const int32_t *__restrict__ tid2eid, int vocab, int T, int E, int k, float scaling,
    int32_t *__restrict__ ids, float *__restrict__ w, float *__restrict__ ssel, int *status) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    const int nw = gridDim.x * kRouteWarps;
    for (int t = gw; t < T; t += nw) {
        int my_id = 0;
        float my_s = 0.0f;
        if (lane < k) {
            int tok = input_ids[t];
            if (tok < 0 || tok >= vocab) {
                record_status(status, MOE_ERR_INVALID_ARG);
                tok = 0;
            }
            int e = tid2eid[(size_t)tok * k + lane];
            if (e < 0 || e >= E) {
                record_status(status, MOE_ERR_INVALID_ARG);
                e = 0;
            }
            my_id = e;
            my_s = sigmoid_exact(z[(size_t)t * E + e]);
        }
        write_weights(t, k, lane, my_id, my_s, scaling, ids, w, ssel);
    }
}

template <int EPL>
void launch_topk(int blocks, cudaStream_t st, const float *z, const float *bias,
                 const uint8_t *vis, int T, int E, int k, float scaling, int32_t *ids, float *w,
                 float *ssel) {
    route_topk_kernel<EPL><<<blocks, kRouteWarps * 32, 0, st>>>(z, bias, vis, T, E, k, scaling,
                                                                ids, w, ssel);
}

}  // namespace

moe_status route_from_logits(const float *logits, const float *bias, const uint8_t *is_vision,
                             const int32_t *input_ids, const int32_t *tid2eid, int vocab, int T,
                             int E, int k, float scaling, moe_route_mode mode, int32_t *ids,
                             float *weights, float *scores_sel, cudaStream_t st) {
    const int want = (T + kRouteWarps - 1) / kRouteWarps;
    const int blocks = want < num_sms() * 16 ? want : num_sms() * 16;
    if (mode == MOE_ROUTE_HASH) {
        int *status = device_status_ptr();
        if (!status) return MOE_ERR_CUDA;
        route_hash_kernel<<<blocks, kRouteWarps * 32, 0, st>>>(
            logits, input_ids, tid2eid, vocab, T, E, k, scaling, ids, weights, scores_sel, status);
    } else {
        const int epl = (E + 31) / 32;
        if (epl <= 1) launch_topk<1>(blocks, st, logits, bias, is_vision, T, E, k, scaling, ids, weights, scores_sel);
        else if (epl <= 2) launch_topk<2>(blocks, st, logits, bias, is_vision, T, E, k, scaling, ids, weights, scores_sel);
        else if (epl <= 4) launch_topk<4>(blocks, st, logits, bias, is_vision, T, E, k, scaling, ids, weights, scores_sel);
        else if (epl <= 8) launch_topk<8>(blocks, st, logits, bias, is_vision, T, E, k, scaling, ids, weights, scores_sel);
        else if (epl <= 12) launch_topk<12>(blocks, st, logits, bias, is_vision, T, E, k, scaling, ids, weights, scores_sel);
        else if (epl <= 16) launch_topk<16>(blocks, st, logits, bias, is_vision, T, E, k, scaling, ids, weights, scores_sel);
        else launch_topk<32>(blocks, st, logits, bias, is_vision, T, E, k, scaling, ids, weights, scores_sel);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace moe

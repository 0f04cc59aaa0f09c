// api.cu -- the C ABI of libmoe (declared in include/moe.h): argument
// validation, workspace carving, the device status word, tensor-map
// encoding, and the order of kernel launches of each entry point.
#include <atomic>
#include <cstring>
#include <initializer_list>
#include <functional>
#include <mutex>

#include "moe_ptx.cuh"
#include "mx_common.cuh"

namespace moe {

// implemented in the other translation units
moe_status route_from_logits(const float *logits, const float *bias, const uint8_t *is_vision,
                             const int32_t *input_ids, const int32_t *tid2eid, int vocab, int T,
                             int E, int k, float scaling, moe_route_mode mode, int32_t *ids,
                             float *weights, float *scores_sel, cudaStream_t st);
bool gate_route_supported(int T, int d, int E, int k);
moe_status launch_gate_route(const uint16_t *x, const uint16_t *Wg, const float *offset,
                             const float *bias, const uint8_t *is_vision,
                             const int32_t *input_ids, const int32_t *tid2eid, int vocab, int T,
                             int d, int E, int k, float scaling, moe_route_mode mode,
                             float *logits, int32_t *ids, float *weights, float *ssel,
                             int32_t *counts, cudaStream_t st);
size_t permute_workspace_bytes(int T, int E, int k);
moe_status launch_permute(const int32_t *ids, const float *weights, const uint16_t *x, int T,
                          int d, int E, int k, int32_t *counts, int32_t *offsets,
                          int32_t *row_token, int32_t *slot_row, float *row_weight,
                          uint16_t *x_perm, void *ws, cudaStream_t st);
size_t dwg_workspace_bytes(int d, int E, long long S);
moe_status launch_combine(const uint16_t *y_perm, const int32_t *slot_row, int T, int d, int k,
                          int with_shared, const float *dz, const int32_t *ids,
                          const uint16_t *Wg, uint16_t *y, cudaStream_t st);
moe_status launch_router_bwd(const float *dw_part, int n_part, const int32_t *slot_row,
                             const int32_t *ids, const float *weights, const float *ssel, int T,
                             int E, int k, float scaling, float *dz_sel, float *dz_row,
                             float *dlogits, float *dweights, cudaStream_t st);
moe_status launch_dwg(const uint16_t *x_perm, const float *dz_row, const int32_t *offsets, int d,
                      int E, long long S, float *part, float *dWg, cudaStream_t st);

namespace {

__device__ int g_status;  // the per-device status word

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDevices];
int g_sms[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

__global__ void wait_timeout_kernel(long long limit, int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing ever arrives on `bar`: the wait must give up on its own
        const WaitCtl wc{&abort_flag, status, limit};
        mbar_wait(&bar, 0, wc);
    }
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace of moe_expert_ffn_backward: [dg|du] and w h (the weight-gradient
// operands), the dw partial sums, and with recompute the g|u of GEMM 1.
struct ExpertBwdWorkspace {
    uint16_t *dGU, *hw;
    float *dw_part, *gu;
    uint8_t *tail_maps;   // weight-gradient scratch (per-group tensor maps, group order)
    size_t bytes;
};

ExpertBwdWorkspace carve_expert_bwd(uint8_t *base, int R, int d, int I, bool recompute) {
    ExpertBwdWorkspace w;
    std::memset(&w, 0, sizeof w);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    w.dGU = reinterpret_cast<uint16_t *>(take((size_t)R * 2 * I * 2));
    w.hw = reinterpret_cast<uint16_t *>(take((size_t)R * I * 2));
    w.dw_part = reinterpret_cast<float *>(take((size_t)R * dgrad2_n_tiles(I) * 4));
    if (recompute) w.gu = reinterpret_cast<float *>(take(((size_t)R + 31) / 32 * 32 * 2 * I * 4));
    w.tail_maps = take(kWgradScratchBytes);
    w.bytes = off;
    (void)d;
    return w;
}

// Workspace of moe_router_backward: dz per slot and per row, dW_g partials.
struct RouterBwdWorkspace {
    float *dz_sel, *dz_row, *dwg_part;
    size_t bytes;
};

RouterBwdWorkspace carve_router_bwd(uint8_t *base, int T, int d, int E, int k) {
    RouterBwdWorkspace w;
    std::memset(&w, 0, sizeof w);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    w.dz_sel = reinterpret_cast<float *>(take((size_t)T * k * 4));
    w.dz_row = reinterpret_cast<float *>(take((size_t)T * k * 4));
    w.dwg_part = reinterpret_cast<float *>(take(dwg_workspace_bytes(d, E, (long long)T * k)));
    w.bytes = off;
    return w;
}

// Workspace of the MX expert backward: [dg|du] in bf16 (dW13) and MX along
// 2I (dgrad 1), w h~ (dW2), the dw partials; with recompute g|u and h~; in
// the layer-level call also x_perm and dY_perm in bf16, dY_perm in MX, dX_perm
// and the router's scratch.
struct MxBwdWorkspace {
    uint16_t *dGU, *hw;
    uint8_t *dGUq, *dGUsf;
    float *dw_part, *gu;
    uint8_t *hq, *hsf;
    uint16_t *x_perm, *dX_perm;
    uint8_t *dYq, *dYsf;
    // the weight gradients' operands, quantised along each group's rows and
    // stored transposed, K-chunk-major (k_chunks chunks of 128 codes and
    // sf_slots 16-byte scale slots per column), and the groups' padded
    // contraction plan
    int32_t *kofs, *sofs;
    // the weight gradients' group order and the run-time tile counter
    int32_t *korder;
    int *tile_counter;
    uint8_t *dYt, *dYtsf, *hwt, *hwtsf, *dGUt, *dGUtsf, *xt, *xtsf;
    int k_chunks, sf_slots;
    RouterBwdWorkspace router;
    size_t bytes;
};

MxBwdWorkspace carve_mx_bwd(uint8_t *base, int G, int R, int d, int I, bool recompute, bool layer,
                            int T, int E, int k) {
    MxBwdWorkspace w;
    std::memset(&w, 0, sizeof w);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    const size_t r = (size_t)R;
    w.dGU = reinterpret_cast<uint16_t *>(take(r * 2 * I * 2));
    w.hw = reinterpret_cast<uint16_t *>(take(r * I * 2));
    w.dGUq = take(r * 2 * I);
    w.dGUsf = take(r * mx_sf_pitch(2 * I));
    w.dw_part = reinterpret_cast<float *>(take(r * mx_dgrad2_n_part(I) * 4));
    // each group's rows padded to a multiple of 128; its scale bytes to 16
    const long long kmax = (long long)R + 127LL * G;
    w.k_chunks = (int)(kmax / 128 + 1);
    w.sf_slots = (int)((kmax / 32 + 16LL * G) / 16 + 1);
    w.kofs = reinterpret_cast<int32_t *>(take((size_t)(G + 1) * 4));
    w.sofs = reinterpret_cast<int32_t *>(take((size_t)(G + 1) * 4));
    w.korder = reinterpret_cast<int32_t *>(take((size_t)(G + 1) * 4));
    w.tile_counter = reinterpret_cast<int *>(take(64));
    const size_t kp = (size_t)w.k_chunks * 128, sp = (size_t)w.sf_slots * 16;
    w.dYt = take((size_t)d * kp);
    w.dYtsf = take((size_t)d * sp);
    w.hwt = take((size_t)I * kp);
    w.hwtsf = take((size_t)I * sp);
    w.dGUt = take((size_t)2 * I * kp);
    w.dGUtsf = take((size_t)2 * I * sp);
    w.xt = take((size_t)d * kp);
    w.xtsf = take((size_t)d * sp);
    if (recompute) {
        w.gu = reinterpret_cast<float *>(take((r + 31) / 32 * 32 * 2 * I * 4));
        w.hq = take(r * I);
        w.hsf = take(r * mx_sf_pitch(I));
    }
    if (layer) {
        w.x_perm = reinterpret_cast<uint16_t *>(take(r * d * 2));
        w.dX_perm = reinterpret_cast<uint16_t *>(take(r * d * 2));
        w.dYq = take(r * d);
        w.dYsf = take(r * mx_sf_pitch(d));
        const RouterBwdWorkspace rw = carve_router_bwd(nullptr, T, d, E, k);
        w.router = carve_router_bwd(take(rw.bytes), T, d, E, k);
    }
    w.bytes = off;
    return w;
}

struct BwdWorkspace {
    uint16_t *dY_perm, *dGU, *hw, *dX_perm, *x_perm;
    float *gu, *dw_part, *dz_sel, *dz_row, *dwg_part;
    uint8_t *tail_maps;   // weight-gradient scratch (per-group tensor maps, group order)
    size_t bytes;
};

BwdWorkspace carve_bwd(uint8_t *base, int T, int d, int E, int k, int I, int flags) {
    BwdWorkspace w;
    std::memset(&w, 0, sizeof w);
    const size_t R = (size_t)T * k + T;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    w.dY_perm = reinterpret_cast<uint16_t *>(take(R * d * 2));
    w.dGU = reinterpret_cast<uint16_t *>(take(R * 2 * I * 2));
    w.hw = reinterpret_cast<uint16_t *>(take(R * I * 2));
    w.dX_perm = reinterpret_cast<uint16_t *>(take(R * d * 2));
    w.dw_part = reinterpret_cast<float *>(take(R * dgrad2_n_tiles(I) * 4));
    w.dz_sel = reinterpret_cast<float *>(take((size_t)T * k * 4));
    w.dz_row = reinterpret_cast<float *>(take((size_t)T * k * 4));
    w.dwg_part = reinterpret_cast<float *>(take(dwg_workspace_bytes(d, E, (long long)T * k)));
    w.tail_maps = take(kWgradScratchBytes);
    if (flags & MOE_FLAG_RECOMPUTE) {
        w.x_perm = reinterpret_cast<uint16_t *>(take(R * d * 2));
        w.gu = reinterpret_cast<float *>(take((R + 31) / 32 * 32 * 2 * I * 4));
    }
    w.bytes = off;
    return w;
}

}  // namespace

int *device_status_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

int num_sms() {
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

static bool encode_2d(CUtensorMap *tm, CUtensorMapDataType dt, const void *base, uint64_t inner,
                      uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner,
                      uint32_t box_outer,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return false;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
    }
    if (!aligned16(base) || (row_pitch_bytes & 15u) != 0 || inner == 0 || outer == 0) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_bf16_2d(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                         uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_2d(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_pitch_bytes,
                     box_inner, box_outer);
}

bool encode_tmap_bf16_2d_sw64(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                              uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_2d(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_pitch_bytes,
                     box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool encode_tmap_f32_2d(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                        uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_2d(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, inner, outer, row_pitch_bytes,
                     box_inner, box_outer);
}

bool encode_tmap_u8_2d(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t outer,
                       uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer,
                       int swizzle_bytes) {
    const CUtensorMapSwizzle swz = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                         : CU_TENSOR_MAP_SWIZZLE_NONE;
    return encode_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner, outer, row_pitch_bytes,
                     box_inner, box_outer, swz);
}

moe_status check_shapes(int T, int d, int E, int k, int I) {
    if (T < 1 || d < 1 || E < 1 || k < 1 || I < 1) return MOE_ERR_INVALID_ARG;
    if (k > E) return MOE_ERR_INVALID_ARG;
    if (k > 32 || E > 1024) return MOE_ERR_UNSUPPORTED;
    if (d % 128 != 0 || I % 64 != 0) return MOE_ERR_UNSUPPORTED;
    const long long R = (long long)T * k + T;
    const long long wide = d > 2 * I ? d : 2 * I;
    if (R * wide >= (1LL << 31) || R >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status launch_selftest_timeout(long long limit, cudaStream_t st) {
    int *status = device_status_ptr();
    if (!status) return MOE_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, st>>>(limit, status);
    return cuda_status(cudaGetLastError());
}

namespace {
std::atomic<int> g_pair_modes{MOE_PAIR_DGRAD2 | MOE_PAIR_WGRAD};
}

int gemm_pair_modes() { return g_pair_modes.load(std::memory_order_relaxed); }

moe_status check_ffn(int G, int max_rows, int d, int I, int S) {
    if (G < 1 || G > 1025 || max_rows < 1 || d < 1 || I < 1 || S < 0) return MOE_ERR_INVALID_ARG;
    if (d % 128 != 0 || I % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)max_rows * (d > 2 * I ? d : 2 * I) >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(int T, int d, int E, int k, int I, int flags) {
    if (check_shapes(T, d, E, k, I) != MOE_OK) return 0;
    size_t b = permute_workspace_bytes(T, E, k);
    // moe_expert_ffn_fused's readiness counters (the calls run one after the
    // other on a stream, so they share the buffer)
    const size_t fc = (size_t)ffn_fused_counters(T * k + T, E + 1) * sizeof(int);
    if (fc > b) b = fc;
    if (flags & MOE_FLAG_BACKWARD) {
        const size_t bw = carve_bwd(nullptr, T, d, E, k, I, flags).bytes;
        if (bw > b) b = bw;
    }
    return b;
}

moe_status moe_route_logits(const float *logits, const float *bias, const uint8_t *is_vision,
                            const int32_t *input_ids, const int32_t *tid2eid, int vocab, int T,
                            int E, int k, float scaling, moe_route_mode mode, int32_t *ids,
                            float *weights, float *scores_sel, void *stream) {
    if (T < 1 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (k > 32 || E > 1024) return MOE_ERR_UNSUPPORTED;
    if (!logits || !ids || !weights || !scores_sel) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_ROUTE_TOPK) {
        if (!bias) return MOE_ERR_INVALID_ARG;
    } else if (mode == MOE_ROUTE_HASH) {
        if (!input_ids || !tid2eid || vocab < 1) return MOE_ERR_INVALID_ARG;
    } else {
        return MOE_ERR_INVALID_ARG;
    }
    return route_from_logits(logits, bias, is_vision, input_ids, tid2eid, vocab, T, E, k,
                             scaling, mode, ids, weights, scores_sel,
                             static_cast<cudaStream_t>(stream));
}

moe_status moe_route(const uint16_t *x, const uint16_t *W_g, const float *logit_offset,
                     const float *bias, const uint8_t *is_vision, const int32_t *input_ids,
                     const int32_t *tid2eid, int vocab, int T, int d, int E, int k,
                     float scaling, moe_route_mode mode, float *logits, int32_t *ids,
                     float *weights, float *scores_sel, void *stream) {
    if (T < 1 || d < 1 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (d % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (!x || !W_g || !logits || !aligned16(x) || !aligned16(W_g) || !aligned16(logits))
        return MOE_ERR_INVALID_ARG;
    if (mode != MOE_ROUTE_TOPK && mode != MOE_ROUTE_HASH) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_ROUTE_TOPK && !bias) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_ROUTE_HASH && (!input_ids || !tid2eid || vocab < 1)) return MOE_ERR_INVALID_ARG;
    if (k > 32 || E > 1024) return MOE_ERR_UNSUPPORTED;
    if (!ids || !weights || !scores_sel) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    moe_status s = launch_gate_gemm(x, W_g, logit_offset, T, d, E, logits, st);
    if (s != MOE_OK) return s;
    return route_from_logits(logits, bias, is_vision, input_ids, tid2eid, vocab, T, E, k,
                             scaling, mode, ids, weights, scores_sel, st);
}

moe_status moe_gate_route(const uint16_t *x, const uint16_t *W_g, const float *logit_offset,
                          const float *bias, const uint8_t *is_vision, const int32_t *input_ids,
                          const int32_t *tid2eid, int vocab, int T, int d, int E, int k,
                          float scaling, moe_route_mode mode, float *logits, int32_t *ids,
                          float *weights, float *scores_sel, int32_t *modality_counts,
                          void *stream) {
    if (T < 1 || d < 1 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (mode != MOE_ROUTE_TOPK && mode != MOE_ROUTE_HASH) return MOE_ERR_INVALID_ARG;
    if (!x || !W_g || !logits || !aligned16(x) || !aligned16(W_g) || !aligned16(logits))
        return MOE_ERR_INVALID_ARG;
    if (mode == MOE_ROUTE_TOPK && !bias) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_ROUTE_HASH && (!input_ids || !tid2eid || vocab < 1)) return MOE_ERR_INVALID_ARG;
    if (!ids || !weights || !scores_sel) return MOE_ERR_INVALID_ARG;
    if (!gate_route_supported(T, d, E, k)) return MOE_ERR_UNSUPPORTED;
    return launch_gate_route(x, W_g, logit_offset, bias, is_vision, input_ids, tid2eid, vocab, T,
                             d, E, k, scaling, mode, logits, ids, weights, scores_sel,
                             modality_counts, static_cast<cudaStream_t>(stream));
}

moe_status moe_permute(const int32_t *ids, const float *weights, const uint16_t *x, int T, int d,
                       int E, int k, int32_t *counts, int32_t *offsets, int32_t *row_token,
                       int32_t *slot_row, float *row_weight, uint16_t *x_perm, void *ws,
                       size_t ws_bytes, void *stream) {
    if (T < 1 || E < 1 || k < 1 || k > E || d < 1) return MOE_ERR_INVALID_ARG;
    if (k > 32 || E > 1024 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k + T >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    if (!ids || !counts || !offsets || !row_token || !slot_row) return MOE_ERR_INVALID_ARG;
    if (row_weight && !weights) return MOE_ERR_INVALID_ARG;
    if (x_perm && (!x || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < permute_workspace_bytes(T, E, k)) return MOE_ERR_WORKSPACE;
    return launch_permute(ids, weights, x, T, d, E, k, counts, offsets, row_token, slot_row,
                          row_weight, x_perm, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                          const uint16_t *W13, const uint16_t *W2, const float *row_weight,
                          int S, int d, int I, float clamp, float *gu_save,
                          uint16_t *h_perm, uint16_t *y_perm, void *ws, size_t ws_bytes,
                          void *stream) {
    (void)ws;
    (void)ws_bytes;
    if (!W2 || !y_perm || !aligned16(W2) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
    moe_status s = check_ffn(G, max_rows, d, I, S);
    if (s != MOE_OK) return s;
    s = moe_expert_gemm1(x_perm, offsets, G, max_rows, W13, d, I, clamp, gu_save, h_perm, stream);
    if (s != MOE_OK) return s;
    return moe_expert_gemm2(h_perm, offsets, G, max_rows, W2, row_weight, S, d, I, y_perm, stream);
}

static moe_status ffn_fused(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                            const uint16_t *W13, const uint16_t *W2, const float *row_weight,
                            int S, int d, int I, float clamp, float *gu_save, uint16_t *h_perm,
                            uint16_t *y_perm, void *ws, size_t ws_bytes, void *stream,
                            int stall_rt, long long wait_limit) {
    moe_status s = check_ffn(G, max_rows, d, I, S);
    if (s != MOE_OK) return s;
    if (I % 128 != 0 || d % 256 != 0) return MOE_ERR_UNSUPPORTED;
    if (!x_perm || !offsets || !W13 || !W2 || !h_perm || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(W13) || !aligned16(W2) || !aligned16(h_perm) ||
        !aligned16(y_perm) || (gu_save && !aligned16(gu_save)))
        return MOE_ERR_INVALID_ARG;
    if (!(clamp > 0.0f)) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < (size_t)ffn_fused_counters(max_rows, G) * sizeof(int) ||
        (reinterpret_cast<uintptr_t>(ws) & 3u) != 0)
        return MOE_ERR_WORKSPACE;
    return launch_ffn12(x_perm, offsets, G, max_rows, W13, W2, row_weight, S, d, I, clamp, h_perm,
                        gu_save, y_perm, static_cast<int *>(ws), static_cast<cudaStream_t>(stream),
                        stall_rt, wait_limit);
}

moe_status moe_expert_ffn_fused(const uint16_t *x_perm, const int32_t *offsets, int G,
                                int max_rows, const uint16_t *W13, const uint16_t *W2,
                                const float *row_weight, int S, int d, int I, float clamp,
                                float *gu_save, uint16_t *h_perm, uint16_t *y_perm, void *ws,
                                size_t ws_bytes, void *stream) {
    return ffn_fused(x_perm, offsets, G, max_rows, W13, W2, row_weight, S, d, I, clamp, gu_save,
                     h_perm, y_perm, ws, ws_bytes, stream, -1, 0);
}

moe_status moe_selftest_ffn_fused_stall(const uint16_t *x_perm, const int32_t *offsets, int G,
                                        int max_rows, const uint16_t *W13, const uint16_t *W2,
                                        const float *row_weight, int S, int d, int I, float clamp,
                                        uint16_t *h_perm, uint16_t *y_perm, void *ws,
                                        size_t ws_bytes, int stall_row_tile,
                                        long long limit_cycles, void *stream) {
    if (stall_row_tile < 0 || limit_cycles <= 0 || limit_cycles >= (1LL << 31))
        return MOE_ERR_INVALID_ARG;
    return ffn_fused(x_perm, offsets, G, max_rows, W13, W2, row_weight, S, d, I, clamp, nullptr,
                     h_perm, y_perm, ws, ws_bytes, stream, stall_row_tile, limit_cycles);
}

int moe_mx_sf_pitch(int K) { return K > 0 ? mx_sf_pitch(K) : 0; }

moe_status moe_mx_quantize(const uint16_t *src, long long rows, int K, uint8_t *q, uint8_t *sf,
                           void *stream) {
    if (rows < 0 || K < 32 || K % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!src || !q || !sf || !aligned16(src) || !aligned16(q) || !aligned16(sf))
        return MOE_ERR_INVALID_ARG;
    return launch_mx_quantize(src, rows, K, q, sf, static_cast<cudaStream_t>(stream));
}

moe_status moe_mx_gather(const uint16_t *x, const int32_t *slot_row, int T, int d, int k,
                         uint8_t *x_perm_q, uint8_t *x_perm_sf, void *stream) {
    if (T < 1 || d < 32 || d % 32 != 0 || k < 1 || k > 32) return MOE_ERR_INVALID_ARG;
    if ((long long)T * (k + 1) * d >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
    if (!x || !slot_row || !x_perm_q || !x_perm_sf || !aligned16(x) || !aligned16(x_perm_q) ||
        !aligned16(x_perm_sf))
        return MOE_ERR_INVALID_ARG;
    return launch_mx_gather(x, slot_row, T, d, k, x_perm_q, x_perm_sf,
                            static_cast<cudaStream_t>(stream));
}

static moe_status check_ffn_mx(int G, int max_rows, int d, int I, int S, float clamp,
                               std::initializer_list<const void *> ptrs, const int32_t *offsets) {
    moe_status s = check_ffn(G, max_rows, d, I, S);
    if (s != MOE_OK) return s;
    if (d % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    for (const void *ptr : ptrs)
        if (!ptr || !aligned16(ptr)) return MOE_ERR_INVALID_ARG;
    if (!offsets || !(clamp > 0.0f)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status moe_expert_gemm1_mx(const uint8_t *x_perm_q, const uint8_t *x_perm_sf,
                               const int32_t *offsets, int G, int max_rows, const uint8_t *W13_q,
                               const uint8_t *W13_sf, int d, int I, float clamp, float *gu_save,
                               uint8_t *h_q, uint8_t *h_sf, void *stream) {
    moe_status s = check_ffn_mx(G, max_rows, d, I, 0, clamp,
                                {x_perm_q, x_perm_sf, W13_q, W13_sf, h_q, h_sf}, offsets);
    if (s != MOE_OK) return s;
    if (gu_save && !aligned16(gu_save)) return MOE_ERR_INVALID_ARG;
    return launch_mx_ffn1(x_perm_q, x_perm_sf, offsets, G, max_rows, W13_q, W13_sf, d, I, clamp,
                          h_q, h_sf, gu_save, static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_gemm2_mx(const uint8_t *h_q, const uint8_t *h_sf, const int32_t *offsets,
                               int G, int max_rows, const uint8_t *W2_q, const uint8_t *W2_sf,
                               const float *row_weight, int S, int d, int I, uint16_t *y_perm,
                               void *stream) {
    moe_status s = check_ffn_mx(G, max_rows, d, I, S, 1.0f, {h_q, h_sf, W2_q, W2_sf, y_perm},
                                offsets);
    if (s != MOE_OK) return s;
    return launch_mx_ffn2(h_q, h_sf, offsets, G, max_rows, W2_q, W2_sf, row_weight, S, d, I, y_perm,
                          static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn_mx(const uint8_t *x_perm_q, const uint8_t *x_perm_sf,
                             const int32_t *offsets, int G, int max_rows, const uint8_t *W13_q,
                             const uint8_t *W13_sf, const uint8_t *W2_q, const uint8_t *W2_sf,
                             const float *row_weight, int S, int d, int I, float clamp,
                             float *gu_save, uint8_t *h_q, uint8_t *h_sf, uint16_t *y_perm,
                             void *stream) {
    moe_status s = check_ffn_mx(G, max_rows, d, I, S, clamp,
                                {x_perm_q, x_perm_sf, W13_q, W13_sf, W2_q, W2_sf, h_q, h_sf,
                                 y_perm}, offsets);
    if (s != MOE_OK) return s;
    s = moe_expert_gemm1_mx(x_perm_q, x_perm_sf, offsets, G, max_rows, W13_q, W13_sf, d, I, clamp,
                            gu_save, h_q, h_sf, stream);
    if (s != MOE_OK) return s;
    return moe_expert_gemm2_mx(h_q, h_sf, offsets, G, max_rows, W2_q, W2_sf, row_weight, S, d, I,
                               y_perm, stream);
}

moe_status moe_mx_quantize_t(const uint16_t *src, int G, int R, int C, uint8_t *q, uint8_t *sf,
                             void *stream) {
    if (G < 1 || C < 1 || R < 32 || R % 32 != 0) return MOE_ERR_INVALID_ARG;
    if ((long long)G * R * C >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
    if (!src || !q || !sf || !aligned16(src) || !aligned16(q) || !aligned16(sf))
        return MOE_ERR_INVALID_ARG;
    return launch_mx_quantize_t(src, G, R, C, q, sf, static_cast<cudaStream_t>(stream));
}

moe_status moe_mx_quantize_both(const uint16_t *src, int G, int R, int C, uint8_t *q,
                                uint8_t *sf, uint8_t *qt, uint8_t *sft, void *stream) {
    if (G < 1 || R < 1 || C < 1) return MOE_ERR_INVALID_ARG;
    if (R % 128 != 0 || C % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)G * R * C >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
    for (const void *p : {static_cast<const void *>(src), static_cast<const void *>(q),
                          static_cast<const void *>(sf), static_cast<const void *>(qt),
                          static_cast<const void *>(sft)})
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    return launch_mx_quantize_both(src, G, R, C, q, sf, qt, sft, static_cast<cudaStream_t>(stream));
}

namespace {

// The expert part of the MX backward on expert-contiguous rows (shared by the
// expert-level and the layer-level call; arguments already checked).
struct MxExpertBwd {
    int G, R, S, d, I;
    float clamp;
    const int32_t *offsets;
    const uint16_t *x_perm;
    const uint8_t *x_perm_q, *x_perm_sf, *W13_q, *W13_sf;
    const float *gu_save;
    const uint8_t *h_q, *h_sf, *W2t_q, *W2t_sf, *W13t_q, *W13t_sf;
    const float *row_weight;
    const uint16_t *dY_rows;      // dY of row r at dY_rows[dY_idx ? dY_idx[r] : r]
    const int32_t *dY_idx;
    const uint8_t *dY_perm_q, *dY_perm_sf;
    uint16_t *dX_perm;
    float *dW13, *dW2;
};

moe_status run_mx_expert_bwd(const MxExpertBwd &a, const MxBwdWorkspace &w, int *n_part,
                             const std::function<bool(int)> &mark, cudaStream_t st) {
    moe_status s;
    const float *gu = a.gu_save;
    const uint8_t *hq = a.h_q, *hsf = a.h_sf;
    if (!mark(MOE_BWD_RECOMPUTE_GEMM1)) return MOE_ERR_CUDA;
    if (!gu) {
        if ((s = launch_mx_ffn1(a.x_perm_q, a.x_perm_sf, a.offsets, a.G, a.R, a.W13_q, a.W13_sf,
                                a.d, a.I, a.clamp, w.hq, w.hsf, w.gu, st)) != MOE_OK)
            return s;
        gu = w.gu;
        hq = w.hq;
        hsf = w.hsf;
    }
    if (!mark(MOE_BWD_DGRAD2)) return MOE_ERR_CUDA;
    if ((s = launch_mx_dgrad2(a.dY_perm_q, a.dY_perm_sf, a.offsets, a.G, a.R, a.W2t_q, a.W2t_sf,
                              gu, hq, hsf, a.row_weight, a.S, a.d, a.I, a.clamp, w.dGU, w.dGUq,
                              w.dGUsf, w.hw, w.dw_part, n_part, w.tile_counter, st)) != MOE_OK)
        return s;
    // the weight gradients in the MX training form: their operands quantised
    // along each group's rows (padded to 128), stored transposed
    if (!mark(MOE_BWD_WGRAD2)) return MOE_ERR_CUDA;
    if ((s = launch_mx_kpad_plan(a.offsets, a.G, w.kofs, w.sofs, st)) != MOE_OK) return s;
    auto rows_t = [&](const uint16_t *src, const int32_t *idx, int C, uint8_t *q, uint8_t *sf) {
        return launch_mx_quantize_rows_t(src, idx, a.offsets, w.kofs, w.sofs, a.G, w.k_chunks, C,
                                         q, sf, st);
    };
    if ((s = rows_t(a.dY_rows, a.dY_idx, a.d, w.dYt, w.dYtsf)) != MOE_OK) return s;
    if ((s = rows_t(w.hw, nullptr, a.I, w.hwt, w.hwtsf)) != MOE_OK) return s;
    if ((s = launch_mx_wgrad(w.dYt, w.dYtsf, w.hwt, w.hwtsf, w.kofs, w.sofs, a.G, a.d, a.I,
                             w.k_chunks, w.sf_slots, a.dW2, w.korder, w.tile_counter, st)) !=
        MOE_OK)
        return s;
    if (!mark(MOE_BWD_DGRAD1)) return MOE_ERR_CUDA;
    // dgrad 1 is MX GEMM 2 with the contraction over 2I and no row weight
    if ((s = launch_mx_ffn2(w.dGUq, w.dGUsf, a.offsets, a.G, a.R, a.W13t_q, a.W13t_sf, nullptr, 0,
                            a.d, 2 * a.I, a.dX_perm, st)) != MOE_OK)
        return s;
    if (!mark(MOE_BWD_WGRAD1)) return MOE_ERR_CUDA;
    if ((s = rows_t(w.dGU, nullptr, 2 * a.I, w.dGUt, w.dGUtsf)) != MOE_OK) return s;
    if ((s = rows_t(a.x_perm, nullptr, a.d, w.xt, w.xtsf)) != MOE_OK) return s;
    return launch_mx_wgrad(w.dGUt, w.dGUtsf, w.xt, w.xtsf, w.kofs, w.sofs, a.G, 2 * a.I, a.d,
                           w.k_chunks, w.sf_slots, a.dW13, w.korder, w.tile_counter, st);
}

}  // namespace

size_t moe_expert_bwd_mx_workspace_size(int G, int max_rows, int d, int I, int recompute) {
    if (G < 1 || G > 1025 || max_rows < 1 || d < 128 || d % 128 != 0 || I < 128 ||
        I % 128 != 0)
        return 0;
    return carve_mx_bwd(nullptr, G, max_rows, d, I, recompute != 0, false, 0, 0, 0).bytes;
}

moe_status moe_expert_ffn_backward_mx(const moe_expert_bwd_mx_args *a, void *stream) {
    if (!a) return MOE_ERR_INVALID_ARG;
    moe_status s = check_ffn_mx(a->G, a->max_rows, a->d, a->I, a->S, a->clamp,
                                {a->x_perm, a->W2t_q, a->W2t_sf, a->W13t_q,
                                 a->W13t_sf, a->dY_perm, a->dY_perm_q, a->dY_perm_sf, a->dX_perm,
                                 a->dW13, a->dW2},
                                a->offsets);
    if (s != MOE_OK) return s;
    if (a->S > a->max_rows) return MOE_ERR_INVALID_ARG;
    if (a->S > 0 && a->dw_rows && !a->row_weight) return MOE_ERR_INVALID_ARG;
    const bool rec = a->gu_save == nullptr;
    const void *need[] = {a->x_perm_q, a->x_perm_sf, a->W13_q, a->W13_sf};
    const void *need_saved[] = {a->gu_save, a->h_q, a->h_sf};
    for (const void *p : need)
        if (rec && (!p || !aligned16(p))) return MOE_ERR_INVALID_ARG;
    for (const void *p : need_saved)
        if (!rec && (!p || !aligned16(p))) return MOE_ERR_INVALID_ARG;
    if (!a->ws ||
        a->ws_bytes < moe_expert_bwd_mx_workspace_size(a->G, a->max_rows, a->d, a->I, rec))
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const MxBwdWorkspace w = carve_mx_bwd(static_cast<uint8_t *>(a->ws), a->G, a->max_rows, a->d,
                                          a->I, rec, false, 0, 0, 0);
    const MxExpertBwd e{a->G, a->max_rows, a->S, a->d, a->I, a->clamp, a->offsets, a->x_perm,
                        a->x_perm_q, a->x_perm_sf, a->W13_q, a->W13_sf, a->gu_save, a->h_q,
                        a->h_sf, a->W2t_q, a->W2t_sf, a->W13t_q, a->W13t_sf, a->row_weight,
                        a->dY_perm, nullptr, a->dY_perm_q, a->dY_perm_sf, a->dX_perm, a->dW13,
                        a->dW2};
    int n_part = 0;
    if ((s = run_mx_expert_bwd(e, w, &n_part, [](int) { return true; }, st)) != MOE_OK) return s;
    if (a->dw_rows && a->S > 0) return launch_row_sum(w.dw_part, a->S, n_part, a->dw_rows, st);
    return MOE_OK;
}

size_t moe_backward_mx_workspace_size(int T, int d, int E, int k, int I, int recompute) {
    if (check_shapes(T, d, E, k, I) != MOE_OK || d % 256 != 0 || I % 128 != 0) return 0;
    const int R = T * k + T;
    return carve_mx_bwd(nullptr, E + 1, R, d, I, recompute != 0, true, T, E, k).bytes;
}

moe_status moe_backward_mx(const moe_bwd_mx_args *a, void *stream) {
    if (!a) return MOE_ERR_INVALID_ARG;
    const int T = a->T, d = a->d, E = a->E, k = a->k, I = a->I;
    moe_status s = check_shapes(T, d, E, k, I);
    if (s != MOE_OK) return s;
    if (d % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    const bool rec = a->gu_save == nullptr;
    const void *need[] = {a->x,        a->W_g,    a->W2t_q,  a->W2t_sf, a->W13t_q, a->W13t_sf,
                          a->ids,      a->weights, a->scores_sel, a->row_weight, a->offsets,
                          a->row_token, a->slot_row, a->dY, a->dX, a->dW_g, a->dW13, a->dW2};
    for (const void *p : need)
        if (!p) return MOE_ERR_INVALID_ARG;
    const void *al[] = {a->x,      a->W_g,    a->W2t_q, a->W2t_sf, a->W13t_q, a->W13t_sf,
                        a->dY,     a->dX,     a->dW_g,  a->dW13,   a->dW2};
    for (const void *p : al)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    const void *need_rec[] = {a->x_perm_q, a->x_perm_sf, a->W13_q, a->W13_sf};
    const void *need_saved[] = {a->gu_save, a->h_q, a->h_sf};
    for (const void *p : need_rec)
        if (rec && (!p || !aligned16(p))) return MOE_ERR_INVALID_ARG;
    for (const void *p : need_saved)
        if (!rec && (!p || !aligned16(p))) return MOE_ERR_INVALID_ARG;
    if (!(a->clamp > 0.0f)) return MOE_ERR_INVALID_ARG;
    if (!a->ws || a->ws_bytes < moe_backward_mx_workspace_size(T, d, E, k, I, rec))
        return MOE_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const std::function<bool(int)> mark = [&](int i) -> bool {
        if (!a->stage_events || !a->stage_events[i]) return true;
        return cudaEventRecord(static_cast<cudaEvent_t>(a->stage_events[i]), st) == cudaSuccess;
    };
    const int S = T * k;
    const int R = S + T;
    const int G = E + 1;
    const MxBwdWorkspace w =
        carve_mx_bwd(static_cast<uint8_t *>(a->ws), G, R, d, I, rec, true, T, E, k);
    // the bf16 rows of x (dW13's operand and dW_g), and the MX rows of dY
    // (dgrad 2); dW2's operand reads dY's rows through row_token
    if (!mark(MOE_BWD_RECOMPUTE_GATHER)) return MOE_ERR_CUDA;
    if ((s = launch_gather_rows(a->x, a->slot_row, T, d, k, w.x_perm, st)) != MOE_OK) return s;
    const MxExpertBwd e{G, R, S, d, I, a->clamp, a->offsets, w.x_perm, a->x_perm_q, a->x_perm_sf,
                        a->W13_q, a->W13_sf, a->gu_save, a->h_q, a->h_sf, a->W2t_q, a->W2t_sf,
                        a->W13t_q, a->W13t_sf, a->row_weight, a->dY, a->row_token, w.dYq,
                        w.dYsf, w.dX_perm, a->dW13, a->dW2};
    // the expert stages mark their own starts; the dY gathers sit between the
    // GEMM-1 recompute and dgrad 2
    const std::function<bool(int)> mark_expert = [&](int i) -> bool {
        if (i == MOE_BWD_DGRAD2) {
            if (!mark(MOE_BWD_GATHER_DY)) return false;
            if (launch_mx_gather(a->dY, a->slot_row, T, d, k, w.dYq, w.dYsf, st) != MOE_OK)
                return false;
        }
        return mark(i);
    };
    int n_part = 0;
    if ((s = run_mx_expert_bwd(e, w, &n_part, mark_expert, st)) != MOE_OK) return s;
    if (!mark(MOE_BWD_ROUTER)) return MOE_ERR_CUDA;
    if ((s = launch_router_bwd(w.dw_part, n_part, a->slot_row, a->ids, a->weights, a->scores_sel,
                               T, E, k, a->scaling, w.router.dz_sel, w.router.dz_row, a->dlogits,
                               a->dweights, st)) != MOE_OK)
        return s;
    if (!mark(MOE_BWD_DX)) return MOE_ERR_CUDA;
    if ((s = launch_combine(w.dX_perm, a->slot_row, T, d, k, 1, w.router.dz_sel, a->ids, a->W_g,
                            a->dX, st)) != MOE_OK)
        return s;
    if (!mark(MOE_BWD_DWG)) return MOE_ERR_CUDA;
    if ((s = launch_dwg(w.x_perm, w.router.dz_row, a->offsets, d, E, (long long)T * k,
                        w.router.dwg_part, a->dW_g,
                        st)) != MOE_OK)
        return s;
    return mark(MOE_BWD_STAGES) ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_expert_gemm1(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                            const uint16_t *W13, int d, int I, float clamp, float *gu_save,
                            uint16_t *h_perm, void *stream) {
    moe_status s = check_ffn(G, max_rows, d, I, 0);
    if (s != MOE_OK) return s;
    if (!x_perm || !offsets || !W13 || !h_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(W13) || !aligned16(h_perm) ||
        (gu_save && !aligned16(gu_save)))
        return MOE_ERR_INVALID_ARG;
    if (!(clamp > 0.0f)) return MOE_ERR_INVALID_ARG;
    return launch_ffn1(x_perm, offsets, G, max_rows, W13, d, I, clamp, h_perm, gu_save,
                       static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_gemm2(const uint16_t *h_perm, const int32_t *offsets, int G, int max_rows,
                            const uint16_t *W2, const float *row_weight, int S, int d, int I,
                            uint16_t *y_perm, void *stream) {
    moe_status s = check_ffn(G, max_rows, d, I, S);
    if (s != MOE_OK) return s;
    if (!h_perm || !offsets || !W2 || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(h_perm) || !aligned16(W2) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
    return launch_ffn2(h_perm, offsets, G, max_rows, W2, row_weight, S, d, I, y_perm,
                       static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const uint16_t *y_perm, const int32_t *slot_row, int T, int d, int k,
                       int with_shared, uint16_t *y, void *stream) {
    if (T < 1 || d < 1 || k < 1) return MOE_ERR_INVALID_ARG;
    if (k > 32 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!y_perm || !slot_row || !y || !aligned16(y_perm) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    return launch_combine(y_perm, slot_row, T, d, k, with_shared, nullptr, nullptr, nullptr, y,
                          static_cast<cudaStream_t>(stream));
}

moe_status moe_backward(const moe_bwd_args *a, void *stream) {
    if (!a) return MOE_ERR_INVALID_ARG;
    const int T = a->T, d = a->d, E = a->E, k = a->k, I = a->I;
    moe_status s = check_shapes(T, d, E, k, I);
    if (s != MOE_OK) return s;
    const bool rec = (a->flags & MOE_FLAG_RECOMPUTE) != 0;
    if ((a->flags & ~MOE_FLAG_RECOMPUTE) != 0) return MOE_ERR_INVALID_ARG;
    if (!a->x || !a->W_g || !a->W13 || !a->W2 || !a->ids || !a->weights || !a->scores_sel ||
        !a->row_weight || !a->offsets || !a->row_token || !a->slot_row || !a->dY || !a->dX ||
        !a->dW_g || !a->dW13 || !a->dW2)
        return MOE_ERR_INVALID_ARG;
    if (!rec && (!a->x_perm || !a->gu_save)) return MOE_ERR_INVALID_ARG;
    const void *al[] = {a->x, a->W_g, a->W13, a->W2, a->dY, a->dX, a->dW_g, a->dW13, a->dW2};
    for (const void *p : al)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!rec && (!aligned16(a->x_perm) || !aligned16(a->gu_save))) return MOE_ERR_INVALID_ARG;
    if (!(a->clamp > 0.0f)) return MOE_ERR_INVALID_ARG;
    const int flags = MOE_FLAG_BACKWARD | (rec ? MOE_FLAG_RECOMPUTE : 0);
    if (!a->ws || a->ws_bytes < moe_workspace_size(T, d, E, k, I, flags)) return MOE_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // profiling hook: an event before each stage and after the last
    auto mark = [&](int i) -> bool {
        if (!a->stage_events || !a->stage_events[i]) return true;
        return cudaEventRecord(static_cast<cudaEvent_t>(a->stage_events[i]), st) == cudaSuccess;
    };
    BwdWorkspace w = carve_bwd(static_cast<uint8_t *>(a->ws), T, d, E, k, I, a->flags);
    const int S = T * k;
    const int R = S + T;
    const int G = E + 1;
    const uint16_t *x_perm = a->x_perm;
    const float *gu = a->gu_save;
    if (!mark(MOE_BWD_RECOMPUTE_GATHER)) return MOE_ERR_CUDA;
    if (rec) {
        // rebuild the permuted input rows and the expert GEMM-1 outputs
        if ((s = launch_gather_rows(a->x, a->slot_row, T, d, k, w.x_perm, st)) != MOE_OK) return s;
    }
    if (!mark(MOE_BWD_RECOMPUTE_GEMM1)) return MOE_ERR_CUDA;
    if (rec) {
        if ((s = launch_ffn1(w.x_perm, a->offsets, G, R, a->W13, d, I, a->clamp, nullptr, w.gu,
                             st)) != MOE_OK)
            return s;
        x_perm = w.x_perm;
        gu = w.gu;
    }
    int n_part = 0;
    if (!mark(MOE_BWD_GATHER_DY)) return MOE_ERR_CUDA;
    if ((s = launch_gather_rows(a->dY, a->slot_row, T, d, k, w.dY_perm, st)) != MOE_OK) return s;
    if (!mark(MOE_BWD_DGRAD2)) return MOE_ERR_CUDA;
    if ((s = launch_dgrad2(w.dY_perm, a->offsets, G, R, a->W2, gu, a->row_weight, S, d, I,
                           a->clamp, w.dGU, w.hw, w.dw_part, &n_part,
                           scratch_tile_counter(w.tail_maps), st)) != MOE_OK)
        return s;
    if (!mark(MOE_BWD_WGRAD2)) return MOE_ERR_CUDA;
    if ((s = launch_wgrad(w.dY_perm, d, w.hw, I, a->offsets, G, R, a->dW2, w.tail_maps, st)) !=
        MOE_OK)
        return s;
    if (!mark(MOE_BWD_DGRAD1)) return MOE_ERR_CUDA;
    if ((s = launch_dgrad1(w.dGU, a->offsets, G, R, a->W13, d, I, w.dX_perm, st)) != MOE_OK)
        return s;
    if (!mark(MOE_BWD_WGRAD1)) return MOE_ERR_CUDA;
    if ((s = launch_wgrad(w.dGU, 2 * I, x_perm, d, a->offsets, G, R, a->dW13, w.tail_maps, st)) !=
        MOE_OK)
        return s;
    if (!mark(MOE_BWD_ROUTER)) return MOE_ERR_CUDA;
    if ((s = launch_router_bwd(w.dw_part, n_part, a->slot_row, a->ids, a->weights, a->scores_sel,
                               T, E, k, a->scaling, w.dz_sel, w.dz_row, a->dlogits, a->dweights,
                               st)) != MOE_OK)
        return s;
    if (!mark(MOE_BWD_DX)) return MOE_ERR_CUDA;
    if ((s = launch_combine(w.dX_perm, a->slot_row, T, d, k, 1, w.dz_sel, a->ids, a->W_g, a->dX,
                            st)) != MOE_OK)
        return s;
    if (!mark(MOE_BWD_DWG)) return MOE_ERR_CUDA;
    if ((s = launch_dwg(x_perm, w.dz_row, a->offsets, d, E, (long long)T * k, w.dwg_part,
                        a->dW_g, st)) != MOE_OK)
        return s;
    return mark(MOE_BWD_STAGES) ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_gather_rows(const void *src, const int32_t *idx, long long n, long long n_src,
                           int row_bytes, void *dst, void *stream) {
    if (n < 0 || n_src < 0 || row_bytes < 4 || row_bytes % 4 != 0) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!idx || !dst || (n_src > 0 && !src)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 3u)
        return MOE_ERR_INVALID_ARG;
    return launch_index_gather(src, idx, n, n_src, row_bytes, dst,
                               static_cast<cudaStream_t>(stream));
}

size_t moe_expert_bwd_workspace_size(int max_rows, int d, int I, int recompute) {
    if (max_rows < 1 || d < 1 || I < 1 || I % 64 != 0) return 0;
    return carve_expert_bwd(nullptr, max_rows, d, I, recompute != 0).bytes;
}

moe_status moe_expert_ffn_backward(const moe_expert_bwd_args *a, void *stream) {
    if (!a) return MOE_ERR_INVALID_ARG;
    moe_status s = check_ffn(a->G, a->max_rows, a->d, a->I, a->S);
    if (s != MOE_OK) return s;
    if (a->S > a->max_rows) return MOE_ERR_INVALID_ARG;
    if (!a->offsets || !a->x_perm || !a->W13 || !a->W2 || !a->dY_perm || !a->dX_perm ||
        !a->dW13 || !a->dW2)
        return MOE_ERR_INVALID_ARG;
    if (a->S > 0 && a->dw_rows && !a->row_weight) return MOE_ERR_INVALID_ARG;
    const void *al[] = {a->x_perm, a->W13, a->W2, a->dY_perm, a->dX_perm, a->dW13, a->dW2};
    for (const void *p : al)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (a->gu_save && !aligned16(a->gu_save)) return MOE_ERR_INVALID_ARG;
    if (!(a->clamp > 0.0f)) return MOE_ERR_INVALID_ARG;
    const bool rec = a->gu_save == nullptr;
    const int R = a->max_rows, d = a->d, I = a->I, G = a->G;
    if (!a->ws || a->ws_bytes < moe_expert_bwd_workspace_size(R, d, I, rec ? 1 : 0))
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ExpertBwdWorkspace w = carve_expert_bwd(static_cast<uint8_t *>(a->ws), R, d, I, rec);
    const float *gu = a->gu_save;
    if (rec) {
        if ((s = launch_ffn1(a->x_perm, a->offsets, G, R, a->W13, d, I, a->clamp, nullptr, w.gu,
                             st)) != MOE_OK)
            return s;
        gu = w.gu;
    }
    int n_part = 0;
    if ((s = launch_dgrad2(a->dY_perm, a->offsets, G, R, a->W2, gu, a->row_weight, a->S, d, I,
                           a->clamp, w.dGU, w.hw, w.dw_part, &n_part,
                           scratch_tile_counter(w.tail_maps), st)) != MOE_OK)
        return s;
    if ((s = launch_wgrad(a->dY_perm, d, w.hw, I, a->offsets, G, R, a->dW2, w.tail_maps, st)) !=
        MOE_OK)
        return s;
    if ((s = launch_dgrad1(w.dGU, a->offsets, G, R, a->W13, d, I, a->dX_perm, st)) != MOE_OK)
        return s;
    if ((s = launch_wgrad(w.dGU, 2 * I, a->x_perm, d, a->offsets, G, R, a->dW13, w.tail_maps,
                          st)) != MOE_OK)
        return s;
    if (a->dw_rows && a->S > 0)
        return launch_row_sum(w.dw_part, a->S, n_part, a->dw_rows, st);
    return MOE_OK;
}

size_t moe_router_bwd_workspace_size(int T, int d, int E, int k) {
    if (T < 1 || d < 1 || E < 1 || k < 1 || k > E) return 0;
    return carve_router_bwd(nullptr, T, d, E, k).bytes;
}

moe_status moe_router_backward(const float *dw_rows, const uint16_t *dX_perm,
                               const uint16_t *x_perm, const int32_t *offsets, const int32_t *ids,
                               const float *weights, const float *scores_sel,
                               const int32_t *slot_row, const uint16_t *W_g, int T, int d, int E,
                               int k, float scaling, uint16_t *dX, float *dlogits,
                               float *dweights, float *dW_g, void *ws, size_t ws_bytes,
                               void *stream) {
    if (T < 1 || d < 1 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (k > 32 || E > 1024 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!dw_rows || !dX_perm || !x_perm || !offsets || !ids || !weights || !scores_sel ||
        !slot_row || !W_g || !dX || !dW_g)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(dX_perm) || !aligned16(x_perm) || !aligned16(W_g) || !aligned16(dX) ||
        !aligned16(dW_g))
        return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < moe_router_bwd_workspace_size(T, d, E, k)) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    RouterBwdWorkspace w = carve_router_bwd(static_cast<uint8_t *>(ws), T, d, E, k);
    moe_status s;
    if ((s = launch_router_bwd(dw_rows, 1, slot_row, ids, weights, scores_sel, T, E, k, scaling,
                               w.dz_sel, w.dz_row, dlogits, dweights, st)) != MOE_OK)
        return s;
    if ((s = launch_combine(dX_perm, slot_row, T, d, k, 1, w.dz_sel, ids, W_g, dX, st)) != MOE_OK)
        return s;
    return launch_dwg(x_perm, w.dz_row, offsets, d, E, (long long)T * k, w.dwg_part, dW_g, st);
}

namespace {

// One forward of the layer described by L from the device rows x into y.
moe_status layer_forward(const moe_layer_buffers *L, const uint16_t *x, uint16_t *y,
                         void *stream) {
    const int T = L->T, d = L->d, E = L->E, k = L->k, I = L->I;
    moe_status s;
    if (L->modality_counts)
        s = moe_gate_route(x, L->W_g, L->logit_offset, L->bias, L->is_vision, L->input_ids,
                           L->tid2eid, L->vocab, T, d, E, k, L->scaling,
                           static_cast<moe_route_mode>(L->mode), L->logits, L->ids, L->weights,
                           L->scores_sel, L->modality_counts, stream);
    else
        s = moe_route(x, L->W_g, L->logit_offset, L->bias, L->is_vision, L->input_ids,
                      L->tid2eid, L->vocab, T, d, E, k, L->scaling,
                      static_cast<moe_route_mode>(L->mode), L->logits, L->ids, L->weights,
                      L->scores_sel, stream);
    if (s != MOE_OK) return s;
    s = moe_permute(L->ids, L->weights, x, T, d, E, k, L->counts, L->offsets, L->row_token,
                    L->slot_row, L->row_weight, L->x_perm, L->ws, L->ws_bytes, stream);
    if (s != MOE_OK) return s;
    const int R = T * k + T;
    s = moe_expert_ffn(L->x_perm, L->offsets, E + 1, R, L->W13, L->W2, L->row_weight, T * k, d,
                       I, L->clamp, (L->flags & MOE_FLAG_RECOMPUTE) ? nullptr : L->gu_save,
                       L->h_perm, L->y_perm, nullptr, 0, stream);
    if (s != MOE_OK) return s;
    return moe_combine(L->y_perm, L->slot_row, T, d, k, 1, y, stream);
}

// The backward of the last forward of L (input rows x) for the upstream
// gradient dY into dX and L's weight gradients.
moe_status layer_backward(const moe_layer_buffers *L, const uint16_t *x, const uint16_t *dY,
                          uint16_t *dX, void *stream) {
    moe_bwd_args a;
    std::memset(&a, 0, sizeof a);
    a.T = L->T; a.d = L->d; a.E = L->E; a.k = L->k; a.I = L->I;
    a.scaling = L->scaling;
    a.clamp = L->clamp;
    a.flags = L->flags & MOE_FLAG_RECOMPUTE;
    a.x = x; a.W_g = L->W_g; a.W13 = L->W13; a.W2 = L->W2;
    a.ids = L->ids; a.weights = L->weights; a.scores_sel = L->scores_sel;
    a.row_weight = L->row_weight; a.offsets = L->offsets; a.row_token = L->row_token;
    a.slot_row = L->slot_row; a.x_perm = L->x_perm; a.gu_save = L->gu_save;
    a.dY = dY; a.dX = dX; a.dW_g = L->dW_g; a.dW13 = L->dW13; a.dW2 = L->dW2;
    a.ws = L->ws; a.ws_bytes = L->ws_bytes;
    return moe_backward(&a, stream);
}

}  // namespace

moe_status moe_layer_step_host(const moe_layer_buffers *L, const uint16_t *x_host,
                               const uint16_t *dY_host, uint16_t *y_host, uint16_t *dX_host,
                               void *stream, void *copy_stream) {
    if (!L || !x_host || !y_host || !L->x || !L->y) return MOE_ERR_INVALID_ARG;
    const bool train = dY_host != nullptr;
    if (train != (dX_host != nullptr)) return MOE_ERR_INVALID_ARG;
    if (train && (!L->dY || !L->dX)) return MOE_ERR_INVALID_ARG;
    moe_status s = check_shapes(L->T, L->d, L->E, L->k, L->I);
    if (s != MOE_OK) return s;
    const size_t row_bytes = (size_t)L->T * L->d * sizeof(uint16_t);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
    const bool overlap = train && cs != nullptr && cs != st;
    // events of this call: the call's start on `stream`, dY uploaded, forward
    // done, y downloaded
    cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
    auto cleanup = [&](moe_status r) {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
        return r;
    };
    if (overlap)
        for (cudaEvent_t &e : ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                return cleanup(MOE_ERR_CUDA);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    if (!ok(cudaMemcpyAsync(L->x, x_host, row_bytes, cudaMemcpyHostToDevice, st)))
        return cleanup(MOE_ERR_CUDA);
    if (overlap) {
        // the upload of dY waits for whatever `stream` ran before this call
        if (!ok(cudaEventRecord(ev[0], st)) || !ok(cudaStreamWaitEvent(cs, ev[0], 0)) ||
            !ok(cudaMemcpyAsync(L->dY, dY_host, row_bytes, cudaMemcpyHostToDevice, cs)) ||
            !ok(cudaEventRecord(ev[1], cs)))
            return cleanup(MOE_ERR_CUDA);
    }
    if ((s = layer_forward(L, L->x, L->y, stream)) != MOE_OK) return cleanup(s);
    if (overlap) {
        if (!ok(cudaEventRecord(ev[2], st)) || !ok(cudaStreamWaitEvent(cs, ev[2], 0)) ||
            !ok(cudaMemcpyAsync(y_host, L->y, row_bytes, cudaMemcpyDeviceToHost, cs)) ||
            !ok(cudaEventRecord(ev[3], cs)) || !ok(cudaStreamWaitEvent(st, ev[1], 0)))
            return cleanup(MOE_ERR_CUDA);
    } else {
        if (!ok(cudaMemcpyAsync(y_host, L->y, row_bytes, cudaMemcpyDeviceToHost, st)))
            return cleanup(MOE_ERR_CUDA);
        if (train &&
            !ok(cudaMemcpyAsync(L->dY, dY_host, row_bytes, cudaMemcpyHostToDevice, st)))
            return cleanup(MOE_ERR_CUDA);
    }
    if (train) {
        if ((s = layer_backward(L, L->x, L->dY, L->dX, stream)) != MOE_OK) return cleanup(s);
        if (!ok(cudaMemcpyAsync(dX_host, L->dX, row_bytes, cudaMemcpyDeviceToHost, st)))
            return cleanup(MOE_ERR_CUDA);
    }
    // `stream` ends after every copy of the step
    if (overlap && !ok(cudaStreamWaitEvent(st, ev[3], 0))) return cleanup(MOE_ERR_CUDA);
    return cleanup(MOE_OK);
}

moe_status moe_layer_steps_host(const moe_layer_buffers *L, const moe_layer_io *second,
                                int n_steps, const uint16_t *const *x_host,
                                const uint16_t *const *dY_host, uint16_t *const *y_host,
                                uint16_t *const *dX_host, void *stream, void *copy_in_stream,
                                void *copy_out_stream) {
    if (!L || !second || n_steps < 0 || !x_host || !y_host) return MOE_ERR_INVALID_ARG;
    if (n_steps == 0) return MOE_OK;
    const bool train = dY_host != nullptr;
    if (train != (dX_host != nullptr)) return MOE_ERR_INVALID_ARG;
    // the two sets of device rows the steps alternate between
    const moe_layer_io io[2] = {{L->x, L->dY, L->y, L->dX}, *second};
    for (const moe_layer_io &b : io) {
        if (!b.x || !b.y || !aligned16(b.x) || !aligned16(b.y)) return MOE_ERR_INVALID_ARG;
        if (train && (!b.dY || !b.dX || !aligned16(b.dY) || !aligned16(b.dX)))
            return MOE_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n_steps; ++i)
        if (!x_host[i] || !y_host[i] || (train && (!dY_host[i] || !dX_host[i])))
            return MOE_ERR_INVALID_ARG;
    moe_status s = check_shapes(L->T, L->d, L->E, L->k, L->I);
    if (s != MOE_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t ci = static_cast<cudaStream_t>(copy_in_stream);
    cudaStream_t co = static_cast<cudaStream_t>(copy_out_stream);
    if (!ci || !co || ci == st || co == st || ci == co) return MOE_ERR_INVALID_ARG;
    const size_t row_bytes = (size_t)L->T * L->d * sizeof(uint16_t);
    // per set: its inputs landed, the step that uses it has finished reading
    // them (backward, or forward without one), its outputs have been read
    // back; and the call's start on `stream`
    cudaEvent_t in_done[2] = {}, used[2] = {}, out_done[2] = {}, fwd_done[2] = {}, start = nullptr;
    auto cleanup = [&](moe_status r) {
        for (int j = 0; j < 2; ++j)
            for (cudaEvent_t e : {in_done[j], used[j], out_done[j], fwd_done[j]})
                if (e) cudaEventDestroy(e);
        if (start) cudaEventDestroy(start);
        return r;
    };
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    for (int j = 0; j < 2; ++j)
        for (cudaEvent_t *e : {&in_done[j], &used[j], &out_done[j], &fwd_done[j]})
            if (!ok(cudaEventCreateWithFlags(e, cudaEventDisableTiming)))
                return cleanup(MOE_ERR_CUDA);
    if (!ok(cudaEventCreateWithFlags(&start, cudaEventDisableTiming))) return cleanup(MOE_ERR_CUDA);
    // the uploads wait for whatever `stream` ran before this call
    if (!ok(cudaEventRecord(start, st)) || !ok(cudaStreamWaitEvent(ci, start, 0)))
        return cleanup(MOE_ERR_CUDA);
    auto upload = [&](int i) {
        const moe_layer_io &b = io[i & 1];
        if (i >= 2 && !ok(cudaStreamWaitEvent(ci, used[i & 1], 0))) return false;
        if (!ok(cudaMemcpyAsync(b.x, x_host[i], row_bytes, cudaMemcpyHostToDevice, ci)))
            return false;
        if (train &&
            !ok(cudaMemcpyAsync(b.dY, dY_host[i], row_bytes, cudaMemcpyHostToDevice, ci)))
            return false;
        return ok(cudaEventRecord(in_done[i & 1], ci));
    };
    if (!upload(0)) return cleanup(MOE_ERR_CUDA);
    for (int i = 0; i < n_steps; ++i) {
        const int j = i & 1;
        const moe_layer_io &b = io[j];
        // step i's inputs are in, and the outputs step i - 2 left in this set
        // have been read back
        if (!ok(cudaStreamWaitEvent(st, in_done[j], 0))) return cleanup(MOE_ERR_CUDA);
        if (i >= 2 && !ok(cudaStreamWaitEvent(st, out_done[j], 0))) return cleanup(MOE_ERR_CUDA);
        if ((s = layer_forward(L, b.x, b.y, stream)) != MOE_OK) return cleanup(s);
        if (!ok(cudaEventRecord(fwd_done[j], st)) || !ok(cudaStreamWaitEvent(co, fwd_done[j], 0)) ||
            !ok(cudaMemcpyAsync(y_host[i], b.y, row_bytes, cudaMemcpyDeviceToHost, co)))
            return cleanup(MOE_ERR_CUDA);
        if (!train && !ok(cudaEventRecord(used[j], st))) return cleanup(MOE_ERR_CUDA);
        // the next step's inputs go up while this step computes
        if (i + 1 < n_steps && !upload(i + 1)) return cleanup(MOE_ERR_CUDA);
        if (train) {
            if ((s = layer_backward(L, b.x, b.dY, b.dX, stream)) != MOE_OK) return cleanup(s);
            if (!ok(cudaEventRecord(used[j], st)) || !ok(cudaStreamWaitEvent(co, used[j], 0)) ||
                !ok(cudaMemcpyAsync(dX_host[i], b.dX, row_bytes, cudaMemcpyDeviceToHost, co)))
                return cleanup(MOE_ERR_CUDA);
        }
        if (!ok(cudaEventRecord(out_done[j], co))) return cleanup(MOE_ERR_CUDA);
    }
    // `stream` ends after every copy of the call
    for (int j = 0; j < 2 && j < n_steps; ++j)
        if (!ok(cudaStreamWaitEvent(st, out_done[j], 0))) return cleanup(MOE_ERR_CUDA);
    if (!ok(cudaStreamWaitEvent(st, in_done[(n_steps - 1) & 1], 0))) return cleanup(MOE_ERR_CUDA);
    return cleanup(MOE_OK);
}

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device-side wait timed out";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

moe_status moe_last_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    int *p = device_status_ptr();
    if (!p) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return MOE_ERR_CUDA;
    return static_cast<moe_status>(v);
}

int moe_set_gemm_pairs(int mask) {
    const int valid = MOE_PAIR_EXPERT_GEMM1 | MOE_PAIR_EXPERT_GEMM2 | MOE_PAIR_DGRAD2 |
                      MOE_PAIR_DGRAD1 | MOE_PAIR_WGRAD;
    return g_pair_modes.exchange(mask & valid);
}

moe_status moe_selftest_wait_timeout(long long limit_cycles, void *stream) {
    if (limit_cycles <= 0 || limit_cycles >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
    return launch_selftest_timeout(limit_cycles, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

/*
 * moe.h -- C ABI of the routed Mixture-of-Experts layer library (libmoe.so).
 *
 * One DeepSeek-V4-style MoE layer on one GPU: gate projection and routing,
 * permutation of token slots into expert-contiguous rows, the two expert
 * matmuls around a clamped SwiGLU, the weighted combine with the shared
 * expert, and the backward of all of it.  Sources (page title, section):
 *
 *   [HP41] "HyperParallel加速DeepSeek-V4.1多模态1M长序列训练", §2.3 MegaKernel:
 *          MegaGate (score, bias ranking, top-k, score extraction,
 *          normalisation and scaling, separate text / vision routing bias,
 *          fused backward of the normalisation chain; the projection matmul
 *          is an ordinary GEMM) and MegaMoE (token dispatch, two expert
 *          matmuls, SwiGLU with the V4.1 clamp, result return).
 *   [HPF]  "MindSpore HyperParallel一键开箱DeepSeek-V4.1-Flash", §01: each MoE
 *          layer has 1 shared and 384 routed experts, 6 active per token.
 *   [TW]   "Twinkle x 昇腾，率先实现Deepseek-V4系列模型高效训练",
 *          "FSDP2-4D并行引擎适配": TopKRouter returns router logits, routing
 *          weights and selected experts; HashRouter looks experts up in
 *          tid2eid[input_ids] and still weights them with the gate logits;
 *          tokens are dispatched to experts, computed, returned and combined
 *          by routing weight.
 *   [TTN]  "DeepSeek-V4昇腾训练支持：基于 CANN 平台的TorchTitan-NPU + AutoFuse
 *          极简训练优化实践", 性能结果与未来展望: FP8 training on MxFP8
 *          low-precision compute as the next step (the MXFP8 calls below).
 *
 * Conventions for every call
 *   - All pointers are DEVICE pointers unless marked [host].  The caller owns
 *     and allocates every buffer, including the workspace; the library never
 *     allocates and never frees.
 *   - bf16 tensors are passed as uint16_t bit patterns.  Every matrix is
 *     row-major and densely packed; base pointers must be 16-byte aligned.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Outputs are overwritten, never accumulated.
 *   - Arguments are validated on the host before anything is launched; a
 *     failure returns MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED and launches
 *     nothing.  A CUDA launch error returns MOE_ERR_CUDA.  Errors found on the
 *     device (an out-of-range table entry, a bounded wait that ran out) are
 *     recorded in a per-device status word read by moe_last_device_status();
 *     kernels never trap.
 *   - Sizes: T tokens, d hidden, E routed experts, k experts per token,
 *     I expert intermediate size, S = T*k routed slots.  Supported: T >= 1,
 *     d % 128 == 0, I % 64 == 0, 1 <= k <= min(E, 32), 1 <= E <= 1024,
 *     (S + T) * max(d, 2I) < 2^31.
 *
 * Shared expert and row space.  The shared expert ([HPF] §01) is group E of
 * the expert weights and runs on every token with weight 1.  Permuted row
 * buffers have S + T rows: rows [0, S) are the routed slots in expert-major
 * order, rows [S, S + T) are the tokens themselves in order (the shared
 * expert's group).  offsets[] therefore has E + 2 entries with
 * offsets[E] = S and offsets[E + 1] = S + T.
 *
 * Expert weights: W13 [E+1, 2I, d] (rows 0..I-1 of each group project to the
 * gate g, rows I..2I-1 to the up value u), W2 [E+1, d, I], gate W_g [E, d].
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size or mode */
    MOE_ERR_UNSUPPORTED = 2,  /* valid but outside the supported shapes */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime or launch error */
    MOE_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up */
    MOE_ERR_WORKSPACE = 5     /* workspace missing or too small */
} moe_status;

typedef enum { MOE_ROUTE_TOPK = 0, MOE_ROUTE_HASH = 1 } moe_route_mode;

/* Flags of moe_workspace_size / moe_backward. */
#define MOE_FLAG_BACKWARD 1   /* size the workspace for moe_backward as well */
#define MOE_FLAG_RECOMPUTE 2  /* backward rebuilds x_perm and g|u instead of reading them */

/* Bytes of workspace that moe_permute, moe_expert_ffn_fused and (with
 * MOE_FLAG_BACKWARD) moe_backward need for these sizes.  One buffer of this
 * size may be reused by every call of one layer; calls on one stream run in
 * order, so reuse is safe.  Returns 0 for unsupported sizes. */
size_t moe_workspace_size(int T, int d, int E, int k, int I, int flags);

/* Gate projection and routing ([HP41] §2.3 MegaGate; [TW] TopKRouter and
 * HashRouter).
 *   logits[t,e] = sum_i x[t,i] W_g[e,i] + logit_offset[e]    fp32, fp32 accumulate
 *   s           = sigmoid(logits)                           (score)
 *   TOPK: key   = fp32(s + bias[m_t, e]), m_t = is_vision[t] ? 1 : 0
 *         ids   = the k largest keys, descending, equal keys by lower id
 *   HASH: ids   = tid2eid[input_ids[t]]  (bias unused)
 *   scores_sel[t,j] = s at ids[t,j]       (unbiased score, fp32 = the sigmoid
 *                                          evaluated in fp64 and rounded once)
 *   weights[t,j]    = scaling * scores_sel[t,j] / sum_j scores_sel[t,j]
 * Arguments
 *   x [T,d] bf16, W_g [E,d] bf16; logit_offset [E] fp32 or NULL (a fixed
 *   per-expert shift, no gradient); bias [2,E] fp32 (row 0 text, row 1
 *   vision); is_vision [T] uint8 or NULL (all text); input_ids [T] int32 and
 *   tid2eid [vocab,k] int32 for HASH (NULL / ignored for TOPK).
 *   Outputs: logits [T,E] fp32 (kept for the backward), ids [T,k] int32,
 *   weights [T,k] fp32, scores_sel [T,k] fp32.
 *   An input id outside [0,vocab) or a table entry outside [0,E) is replaced
 *   by 0 and recorded as MOE_ERR_INVALID_ARG in the device status word. */
moe_status moe_route(const uint16_t *x, const uint16_t *W_g, const float *logit_offset,
                     const float *bias, const uint8_t *is_vision, const int32_t *input_ids,
                     const int32_t *tid2eid, int vocab, int T, int d, int E, int k,
                     float scaling, moe_route_mode mode, float *logits, int32_t *ids,
                     float *weights, float *scores_sel, void *stream);

/* Routing only, from given logits (the MegaGate pipeline without the
 * projection, [HP41] §2.3).  Same semantics and outputs as moe_route. */
moe_status moe_route_logits(const float *logits, const float *bias, const uint8_t *is_vision,
                            const int32_t *input_ids, const int32_t *tid2eid, int vocab, int T,
                            int E, int k, float scaling, moe_route_mode mode, int32_t *ids,
                            float *weights, float *scores_sel, void *stream);

/* Gate projection and routing in one kernel, with the expert load of each
 * modality ([HP41] §2.3 MegaGate; [HP41] §01 item 5, native multimodal MoE:
 * text and vision load are balanced separately).  Same semantics and outputs
 * as moe_route, plus
 *   modality_counts [2,E] int32 or NULL: modality_counts[m,e] = number of
 *   slots (t,j) with ids[t,j] = e and m = is_vision[t] ? 1 : 0 (row 0 text,
 *   row 1 vision); rows sum to T*k.  Overwritten (zeroed on `stream` first).
 * The logits of each 128-token block stay in tensor memory (of one CTA, or
 * split by experts over a pair of CTAs when E % 64 == 0) and are routed
 * there: they are written once, and only the few logits within each token's
 * selection window (its whole row when many keys tie) are read back.
 * Supported: d % 64 == 0, E % 32 == 0, 32 <= E <= 512, 1 <= k <= min(8, E);
 * other sizes return MOE_ERR_UNSUPPORTED (use moe_route).  Needs logits 16-
 * byte aligned; ids, weights, scores_sel and modality_counts 4-byte aligned. */
moe_status moe_gate_route(const uint16_t *x, const uint16_t *W_g, const float *logit_offset,
                          const float *bias, const uint8_t *is_vision, const int32_t *input_ids,
                          const int32_t *tid2eid, int vocab, int T, int d, int E, int k,
                          float scaling, moe_route_mode mode, float *logits, int32_t *ids,
                          float *weights, float *scores_sel, int32_t *modality_counts,
                          void *stream);

/* Token dispatch on one GPU ([HP41] §2.3 MegaMoE "token dispatch"; [TW]
 * FSDP2-4D: selected experts become global expert ids of one dispatch).
 * Stable expert-major permutation of the S = T*k slots (expert, then token,
 * then slot), plus the shared expert's identity rows:
 *   counts [E]        slots per routed expert
 *   offsets [E+2]     first row of each group; offsets[E] = S, offsets[E+1] = S+T
 *   row_token [S+T]   token of each row (rows >= S: row - S)
 *   slot_row [S]      row of slot j of token t at index t*k + j
 *   row_weight [S]    weights[t,j] moved to its row (NULL: not produced; needs
 *                     weights [T,k] fp32)
 *   x_perm [S+T, d]   x_perm[row] = x[row_token[row]] (NULL: indices only)
 * ids [T,k] int32 must lie in [0,E) (out-of-range ids are recorded as
 * MOE_ERR_INVALID_ARG on the device and their slots are left unwritten).
 * Needs d % 8 == 0 when x_perm is given.
 * Workspace: moe_workspace_size(T,d,E,k,I,0) bytes. */
moe_status moe_permute(const int32_t *ids, const float *weights, const uint16_t *x, int T, int d,
                       int E, int k, int32_t *counts, int32_t *offsets, int32_t *row_token,
                       int32_t *slot_row, float *row_weight, uint16_t *x_perm, void *ws,
                       size_t ws_bytes, void *stream);

/* moe_permute without a workspace argument: the same dispatch with the same
 * outputs, for callers that cannot allocate device memory -- for instance a
 * plugin running inside a host program that owns every device allocation, or
 * a runtime that forbids allocation once it is running so that latency stays
 * predictable.  The pages have no counterpart of this call; it exists only for
 * such callers.
 * Its scratch memory is one fixed array inside the library (4 MiB per GPU that
 * loads the library, held until the process exits), enough for
 * ceil(T*k / 256) * E <= 1048576 -- e.g. T = 65536, k = 6, E = 384.  Larger
 * sizes return MOE_ERR_UNSUPPORTED and launch nothing.  The call itself
 * allocates nothing.  The first call on a device looks up the array's device
 * address (a CUDA runtime query, done once per device); under lazy module
 * loading (the CUDA default) that first query may also load the library's
 * module on that device and so reserve the array's 4 MiB at that moment.
 * Make that first call during set-up, before any stream capture and before
 * the point from which the program forbids allocation.  All calls share the one array: two calls whose
 * kernels overlap on the GPU (different streams, different host threads) race
 * and give wrong results; calls in order on one stream are safe. */
moe_status moe_permute_noalloc(const int32_t *ids, const float *weights, const uint16_t *x, int T,
                               int d, int E, int k, int32_t *counts, int32_t *offsets,
                               int32_t *row_token, int32_t *slot_row, float *row_weight,
                               uint16_t *x_perm, void *stream);

/* The expert FFN on expert-contiguous rows ([HP41] §2.3 MegaMoE: two expert
 * matmuls around SwiGLU with clamp; [HPF] §01 shared expert as group E).
 * For every group g < G and row r in [offsets[g], offsets[g+1]):
 *   [g | u]  = x_perm[r] W13[g]^T                      (fp32 accumulate)
 *   h[r]     = bf16( silu(min(g, clamp)) * clamp(u, -clamp, clamp) )
 *   y[r]     = bf16( row_weight[r] * (h[r] W2[g]^T) )  (row_weight = 1 for r >= S
 *                                                       or when NULL)
 * Arguments: x_perm [R,d] bf16 with R = offsets[G]; offsets [G+1] int32
 * (device; e.g. the E+2 offsets of moe_permute with G = E+1); W13 [G,2I,d],
 * W2 [G,d,I] bf16; row_weight [S] fp32 or NULL; S = rows carrying a routing
 * weight.  Outputs h_perm [R,I] bf16, y_perm [R,d] bf16, and gu_save (when
 * not NULL): the fp32 GEMM-1 accumulators g (columns 0..I-1) and u (columns
 * I..2I-1), kept for the backward, which recomputes h from them bit for bit.
 * gu_save holds ceil(R/32)*32 x 2I floats in blocks of 32 rows: element
 * (r, c) is at ((r/32)*(I/2) + c/4)*128 + (r%32)*4 + c%4 (row-block
 * interleaved, so that 32 rows are read and written in contiguous runs).  max_rows is an upper
 * bound of R known on the host (sizes the launch; S + T for a full layer).
 * Workspace: none is needed (ws may be NULL). */
moe_status moe_expert_ffn(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                          const uint16_t *W13, const uint16_t *W2, const float *row_weight,
                          int S, int d, int I, float clamp, float *gu_save,
                          uint16_t *h_perm, uint16_t *y_perm, void *ws, size_t ws_bytes,
                          void *stream);

/* The same two expert matmuls as moe_expert_ffn in ONE persistent launch
 * ([HP41] §2.3 MegaMoE: the two expert matmuls and the SwiGLU with the V4.1
 * clamp organised as one fused chain, linked by tile-level dependencies).
 * The tiles of the first matmul come first in a static schedule over all
 * SMs; a tile of the second matmul waits, in the kernel, until every tile of
 * the first that writes its 128 rows of h has finished (per-row-tile
 * counters in `ws`), so the second matmul starts on early row tiles while the
 * first is still finishing the last ones, without a second launch.
 * Arguments and outputs as moe_expert_ffn; h_perm is required (it carries h
 * between the two matmuls).  ws: at least 4 * (ceil(max_rows/128) + G) bytes,
 * 4-byte aligned (moe_workspace_size covers it), zeroed by the call itself.
 * Supported: I % 128 == 0 and d % 256 == 0, else MOE_ERR_UNSUPPORTED.  The
 * waits assume the whole grid is resident (one CTA per SM, nothing else
 * running on the GPU's SMs); a wait that runs out ends the kernel and
 * records MOE_ERR_TIMEOUT in the device status word. */
moe_status moe_expert_ffn_fused(const uint16_t *x_perm, const int32_t *offsets, int G,
                                int max_rows, const uint16_t *W13, const uint16_t *W2,
                                const float *row_weight, int S, int d, int I, float clamp,
                                float *gu_save, uint16_t *h_perm, uint16_t *y_perm, void *ws,
                                size_t ws_bytes, void *stream);

/* The two halves of moe_expert_ffn, for callers that schedule them apart.
 * moe_expert_gemm1 writes h_perm (and gu_save when not NULL);
 * moe_expert_gemm2 reads h_perm and writes y_perm.  Same arguments, layouts
 * and rules as moe_expert_ffn. */
moe_status moe_expert_gemm1(const uint16_t *x_perm, const int32_t *offsets, int G, int max_rows,
                            const uint16_t *W13, int d, int I, float clamp, float *gu_save,
                            uint16_t *h_perm, void *stream);
moe_status moe_expert_gemm2(const uint16_t *h_perm, const int32_t *offsets, int G, int max_rows,
                            const uint16_t *W2, const float *row_weight, int S, int d, int I,
                            uint16_t *y_perm, void *stream);

/* Result return and weighted combine ([HP41] §2.3 MegaMoE "result return";
 * [TW] combine by routing weight).  Gather form, no atomics, fixed order:
 *   y[t] = bf16( y_perm[S + t] + sum_{j<k} y_perm[slot_row[t*k + j]] )   (fp32 sums)
 * y_perm [S+T,d] bf16 already carries the routing weights; pass
 * with_shared = 0 to leave out the shared rows. */
moe_status moe_combine(const uint16_t *y_perm, const int32_t *slot_row, int T, int d, int k,
                       int with_shared, uint16_t *y, void *stream);

/* Everything moe_backward reads and writes.  Forward state is what the
 * forward calls above returned. */
typedef struct {
    int T, d, E, k, I;
    float scaling, clamp;
    int flags;                    /* MOE_FLAG_RECOMPUTE or 0 */
    /* forward inputs */
    const uint16_t *x;            /* [T,d] */
    const uint16_t *W_g;          /* [E,d] */
    const uint16_t *W13;          /* [E+1,2I,d] */
    const uint16_t *W2;           /* [E+1,d,I] */
    /* saved forward state */
    const int32_t *ids;           /* [T,k] */
    const float *weights;         /* [T,k] */
    const float *scores_sel;      /* [T,k] */
    const float *row_weight;      /* [S] (moe_permute) */
    const int32_t *offsets;       /* [E+2] */
    const int32_t *row_token;     /* [S+T] */
    const int32_t *slot_row;      /* [S] */
    const uint16_t *x_perm;       /* [S+T,d]; ignored with MOE_FLAG_RECOMPUTE */
    const float *gu_save;         /* moe_expert_ffn's gu_save; ignored with MOE_FLAG_RECOMPUTE */
    /* upstream gradient */
    const uint16_t *dY;           /* [T,d] */
    /* outputs (overwritten) */
    uint16_t *dX;                 /* [T,d] bf16 */
    float *dW_g;                  /* [E,d] fp32 */
    float *dW13;                  /* [E+1,2I,d] fp32 */
    float *dW2;                   /* [E+1,d,I] fp32 */
    float *dlogits;               /* [T,E] fp32 or NULL (zero off the selection) */
    float *dweights;              /* [T,k] fp32 or NULL (gradient of the routing weights) */
    void *ws;                     /* moe_workspace_size(..., MOE_FLAG_BACKWARD | flags) bytes */
    size_t ws_bytes;
    /* [host] profiling hook, or NULL: MOE_BWD_STAGES + 1 cudaEvent_t handles
     * (created by the caller); event i is recorded on `stream` before stage i
     * and the last one after the last stage, so the caller can time each stage
     * with cudaEventElapsedTime.  A NULL entry is skipped. */
    void *const *stage_events;
} moe_bwd_args;

/* Stages of moe_backward, in launch order (the two recompute stages are
 * empty without MOE_FLAG_RECOMPUTE). */
enum {
    MOE_BWD_RECOMPUTE_GATHER = 0,  /* x_perm rebuilt from x */
    MOE_BWD_RECOMPUTE_GEMM1 = 1,   /* g|u rebuilt (expert GEMM 1) */
    MOE_BWD_GATHER_DY = 2,         /* dY_perm */
    MOE_BWD_DGRAD2 = 3,            /* dA = dY_perm W2, SwiGLU backward, dw */
    MOE_BWD_WGRAD2 = 4,            /* dW2 */
    MOE_BWD_DGRAD1 = 5,            /* dX_perm = [dg|du] W13 */
    MOE_BWD_WGRAD1 = 6,            /* dW13 */
    MOE_BWD_ROUTER = 7,            /* routing-weight chain -> dz */
    MOE_BWD_DX = 8,                /* dX assembly with the gate term */
    MOE_BWD_DWG = 9,               /* dW_g */
    MOE_BWD_STAGES = 10
};

/* Backward of the whole layer (analytic chain rule of the forward above;
 * [HP41] §2.3 names the fused backward of MegaGate's normalisation chain).
 *   dY_perm[r] = dY[row_token[r]]
 *   dA         = dY_perm W2[g]                 dw[r] = <h[r], dA>
 *   dH = w dA;  dg = dH clamp(u) silu'(min(g,c)) [g <= c];  du = dH silu(min(g,c)) [|u| <= c]
 *   dW2[g]  = sum_r dY_perm[r]^T (w h)[r]      dW13[g] = sum_r [dg|du][r]^T x_perm[r]
 *   dX_perm = [dg|du] W13[g]
 *   ds_j = (scaling dw_j - sum_i dw_i w_i) / S_t,  dz_j = ds_j s_j (1 - s_j)
 *   dX[t] = dX_perm[S+t] + sum_j dX_perm[slot_row[t,j]] + sum_j dz_j W_g[ids_j]
 *   dW_g  = dz^T x
 * The bias gets no gradient (it only ranks); hash routing has the same
 * weight chain.  Clamp gradients pass where the argument equals the bound. */
moe_status moe_backward(const moe_bwd_args *args, void *stream);

/* ------------------------------------------- expert parallelism pieces
 * With the experts split over GPUs ("Twinkle x 昇腾…", FSDP2-4D: dispatch to
 * the expert's owner, local expert compute, all-to-all back, combine by
 * routing weight), the caller's collective moves permuted rows between ranks
 * and the calls below do each rank's share: moe_gather_rows regroups rows
 * around an exchange, moe_expert_ffn (forward) and moe_expert_ffn_backward
 * run on the rows a rank's experts received, and moe_router_backward
 * finishes the backward on the rank that routed the tokens. */

/* dst row i = src row idx[i] for i < n (rows of row_bytes bytes, a multiple
 * of 4; 16-byte rows with 16-byte aligned src and dst move as vectors).  A
 * negative idx[i] writes a zero row; idx[i] >= n_src is recorded as
 * MOE_ERR_INVALID_ARG in the device status word and leaves row i unwritten.
 * src [n_src rows], idx int32 [n], dst [n rows]; 4-byte aligned. */
moe_status moe_gather_rows(const void *src, const int32_t *idx, long long n, long long n_src,
                           int row_bytes, void *dst, void *stream);

/* Backward of moe_expert_ffn on its rows (the same four matmuls and clamped
 * SwiGLU backward as in moe_backward, without the routing or combine):
 *   dA = dY_perm[r] W2[g];  dw_rows[r] = <h[r], dA>  (r < S)
 *   dH = w dA;  [dg|du] as in moe_backward;  dX_perm[r] = [dg|du] W13[g]
 *   dW2[g] = sum_r dY_perm[r]^T (w h)[r];  dW13[g] = sum_r [dg|du][r]^T x_perm[r]
 * for every group g < G and row r in [offsets[g], offsets[g+1]), w = row_weight[r]
 * for r < S (rows >= S carry weight 1, e.g. the shared expert's).  gu_save:
 * moe_expert_ffn's saved g|u of these rows, or NULL to recompute it from
 * x_perm into the workspace.  Outputs are overwritten.  Workspace:
 * moe_expert_bwd_workspace_size(max_rows, d, I, gu_save == NULL). */
typedef struct {
    int G, max_rows, S, d, I;
    float clamp;
    const int32_t *offsets;       /* [G+1] */
    const uint16_t *x_perm;       /* [R,d] the rows' GEMM-1 input */
    const uint16_t *W13;          /* [G,2I,d] */
    const uint16_t *W2;           /* [G,d,I] */
    const float *row_weight;      /* [S] or NULL (weight 1) */
    const float *gu_save;         /* or NULL: recompute */
    const uint16_t *dY_perm;      /* [R,d] gradient at the rows' outputs */
    uint16_t *dX_perm;            /* [R,d] out */
    float *dw_rows;               /* [S] out or NULL */
    float *dW13;                  /* [G,2I,d] fp32 out */
    float *dW2;                   /* [G,d,I] fp32 out */
    void *ws;
    size_t ws_bytes;
} moe_expert_bwd_args;
size_t moe_expert_bwd_workspace_size(int max_rows, int d, int I, int recompute);
moe_status moe_expert_ffn_backward(const moe_expert_bwd_args *args, void *stream);

/* The routing and combine part of moe_backward, on the rank that routed the
 * tokens: from the routing-weight gradient of each routed row (dw_rows [S],
 * indexed by permuted row) and the input gradient of every permuted row
 * (dX_perm [S+T,d], the routed rows in this rank's permuted order, then the
 * shared expert's), the normalisation-chain backward (dz, as in
 * moe_backward), dX = dX_perm[S+t] + sum_j dX_perm[slot_row[t,j]] + dz W_g,
 * and dW_g = dz^T x (from this rank's x_perm and offsets).  dlogits /
 * dweights as in moe_backward (nullable).  Workspace:
 * moe_router_bwd_workspace_size(T,d,E,k). */
size_t moe_router_bwd_workspace_size(int T, int d, int E, int k);
moe_status moe_router_backward(const float *dw_rows, const uint16_t *dX_perm,
                               const uint16_t *x_perm, const int32_t *offsets, const int32_t *ids,
                               const float *weights, const float *scores_sel,
                               const int32_t *slot_row, const uint16_t *W_g, int T, int d, int E,
                               int k, float scaling, uint16_t *dX, float *dlogits,
                               float *dweights, float *dW_g, void *ws, size_t ws_bytes,
                               void *stream);

/* ------------------------------------------------- whole layer from host
 * One layer as everything a training step touches: its sizes and options,
 * its weights and routing inputs, and every device buffer of the calls above
 * (all allocated by the caller, as for those calls). */
typedef struct {
    int T, d, E, k, I;
    float scaling, clamp;
    int flags;                    /* MOE_FLAG_RECOMPUTE or 0 */
    int mode;                     /* moe_route_mode */
    const uint16_t *W_g;          /* [E,d] */
    const uint16_t *W13;          /* [E+1,2I,d] */
    const uint16_t *W2;           /* [E+1,d,I] */
    const float *logit_offset;    /* [E] or NULL */
    const float *bias;            /* [2,E] (top-k mode; row 0 text, row 1 vision) */
    const uint8_t *is_vision;     /* [T] or NULL */
    const int32_t *input_ids;     /* [T] (hash mode) */
    const int32_t *tid2eid;       /* [vocab,k] (hash mode) */
    int vocab;
    /* device copies of the step's host input and output rows, [T,d] bf16 each */
    uint16_t *x, *y, *dY, *dX;    /* dY and dX may be NULL for forward-only steps */
    /* forward state (moe_gate_route / moe_route, moe_permute, moe_expert_ffn) */
    float *logits;                /* [T,E] */
    int32_t *ids;                 /* [T,k] */
    float *weights, *scores_sel;  /* [T,k] */
    int32_t *modality_counts;     /* [2,E]: route with moe_gate_route; NULL: with moe_route */
    int32_t *counts;              /* [E] */
    int32_t *offsets;             /* [E+2] */
    int32_t *row_token;           /* [S+T] */
    int32_t *slot_row;            /* [S] */
    float *row_weight;            /* [S] */
    uint16_t *x_perm, *h_perm, *y_perm; /* [S+T,d], [S+T,I], [S+T,d] */
    float *gu_save;               /* as for moe_expert_ffn; NULL with MOE_FLAG_RECOMPUTE */
    /* gradients (training steps) */
    float *dW_g, *dW13, *dW2;
    void *ws;                     /* moe_workspace_size(T,d,E,k,I, MOE_FLAG_BACKWARD | flags) */
    size_t ws_bytes;
} moe_layer_buffers;

/* One step of the layer from and to HOST memory: x_host is copied to L->x,
 * the forward runs (routing, dispatch, both expert matmuls, combine into
 * L->y) and L->y is copied to y_host; with dY_host, dY_host is copied to
 * L->dY, the backward runs (moe_backward into L->dX and the weight
 * gradients) and L->dX is copied to dX_host.  All four host arrays are
 * [host] [T,d] bf16; dY_host and dX_host are both NULL (forward only) or
 * both given.  Copies are cudaMemcpyAsync: host memory should be page-locked
 * for them to run asynchronously.  With copy_stream (a second cudaStream_t)
 * the upload of dY overlaps the forward and the download of y overlaps the
 * backward; the call still leaves `stream` waiting for every copy, so work
 * queued on `stream` afterwards sees the step complete (the call creates and
 * releases a few CUDA events; it allocates no memory).  Returns the first
 * failing call's status. */
moe_status moe_layer_step_host(const moe_layer_buffers *L, const uint16_t *x_host,
                               const uint16_t *dY_host, uint16_t *y_host, uint16_t *dX_host,
                               void *stream, void *copy_stream);

/* A second set of the layer's device rows ([T,d] bf16 each; dY and dX NULL
 * for forward-only steps). */
typedef struct {
    uint16_t *x, *dY, *y, *dX;
} moe_layer_io;

/* n_steps steps of the layer from and to HOST memory, pipelined: step i
 * copies x_host[i] (and dY_host[i]) in and y_host[i] (and dX_host[i]) out,
 * as moe_layer_step_host, with the steps alternating between L's device rows
 * and `second`, so that step i + 1's uploads (on copy_in_stream) and step i's
 * downloads (on copy_out_stream) overlap the neighbouring steps' compute on
 * `stream`.  Three distinct streams; the pointer arrays hold n_steps host
 * buffers each (page-locked for asynchronous copies; dY_host and dX_host both
 * NULL for forward-only steps).  The results are those of n_steps calls of
 * moe_layer_step_host (the weight gradients are the last step's).  `stream`
 * ends after every copy of the call; it creates and releases a few CUDA
 * events and allocates no memory.  Returns the first failing call's status. */
moe_status moe_layer_steps_host(const moe_layer_buffers *L, const moe_layer_io *second,
                                int n_steps, const uint16_t *const *x_host,
                                const uint16_t *const *dY_host, uint16_t *const *y_host,
                                uint16_t *const *dX_host, void *stream, void *copy_in_stream,
                                void *copy_out_stream);

/* ---------------------------------------------------------------- MXFP8
 * Low-precision expert matmuls ([TTN] outlook: FP8 training on MxFP8
 * compute).  The pages fix no format; these calls use the OCP Microscaling
 * Formats (MX) v1.0 specification with FP8 E4M3 elements:
 *   - a block is 32 consecutive elements along the contraction dimension
 *     (a row of a K-major matrix), with one E8M0 scale code c: X = 2^(c-127);
 *   - element codes are OCP E4M3 (bias 7, no infinities, largest 448);
 *   - quantisation: X = 2^(floor(log2 max|v|) - 8), exponent clamped to
 *     [-127, 127] (code 0 for an all-zero block); element = v / X rounded to
 *     the nearest E4M3 value, ties to even, saturated at +-448, the sign kept
 *     for values that round to zero.
 * A quantised [rows, K] matrix is a pair of byte arrays:
 *   q  [rows, K]                 E4M3 codes, row-major (pitch K bytes)
 *   sf [rows, moe_mx_sf_pitch(K)] E8M0 codes, block b of row r at
 *                                sf[r * pitch + b]; the padding bytes of a row
 *                                are neither read for results nor written.
 * Both must be 16-byte aligned; K % 32 == 0.  The MX expert matmuls compute
 * with the exact values of the operands (an E4M3 value times its scale is
 * exact in bf16; products accumulate in fp32), so they differ from a
 * block-scaled MMA only in the order of the fp32 additions.  Operand blocks
 * with scales below 2^-117 are outside that exactness. */

/* Bytes per row of the scale array for a contraction of K elements: K/32
 * rounded up to a multiple of 16. */
int moe_mx_sf_pitch(int K);

/* MX quantisation of a bf16 [rows, K] matrix along its rows (weights once at
 * load time: W13 as [G*2I, d], W2 as [G*d, I]).  Needs K % 32 == 0, rows >= 0;
 * src, q and sf 16-byte aligned, else MOE_ERR_INVALID_ARG. */
moe_status moe_mx_quantize(const uint16_t *src, long long rows, int K, uint8_t *q, uint8_t *sf,
                           void *stream);

/* Dispatch gather into MX rows ([HP41] §2.3 MegaMoE token dispatch): each
 * token row x[t] (bf16 [T, d]) is quantised once and written to rows
 * slot_row[t*k + j] (j < k) and S + t of x_perm_q [S+T, d] / x_perm_sf
 * [S+T, moe_mx_sf_pitch(d)], S = T*k; slot_row comes from moe_permute (which
 * is called with x = NULL for the indices alone).  Needs d % 32 == 0. */
moe_status moe_mx_gather(const uint16_t *x, const int32_t *slot_row, int T, int d, int k,
                         uint8_t *x_perm_q, uint8_t *x_perm_sf, void *stream);

/* MXFP8 expert FFN on expert-contiguous rows: the computation of
 * moe_expert_ffn with MX operands.  For every group g < G and row r in
 * [offsets[g], offsets[g+1]):
 *   [g | u] = x~[r] W13~[g]^T                  (exact products, fp32 sums)
 *   h~[r]   = MX( silu(min(g, clamp)) * clamp(u, -clamp, clamp) )  along I
 *   y[r]    = bf16( row_weight[r] * (h~[r] W2~[g]^T) )
 * x~ = (x_perm_q, x_perm_sf) [R, d]; W13~ = (W13_q, W13_sf) [G*2I, d];
 * W2~ = (W2_q, W2_sf) [G*d, I]; row_weight [S] fp32 or NULL (1 for rows >= S).
 * Outputs: h_q [R, I] and h_sf [R, moe_mx_sf_pitch(I)] (the MX h), y_perm
 * [R, d] bf16.  max_rows bounds R = offsets[G] (sizes the launch).  Needs
 * d % 256 == 0 and I % 128 == 0 (else MOE_ERR_UNSUPPORTED), clamp > 0 and
 * 16-byte aligned arrays (else MOE_ERR_INVALID_ARG).  No workspace. */
moe_status moe_expert_ffn_mx(const uint8_t *x_perm_q, const uint8_t *x_perm_sf,
                             const int32_t *offsets, int G, int max_rows, const uint8_t *W13_q,
                             const uint8_t *W13_sf, const uint8_t *W2_q, const uint8_t *W2_sf,
                             const float *row_weight, int S, int d, int I, float clamp,
                             float *gu_save, uint8_t *h_q, uint8_t *h_sf, uint16_t *y_perm,
                             void *stream);

/* The two matmuls of moe_expert_ffn_mx as separate calls (same arguments
 * and checks; GEMM 1 writes h_q / h_sf, GEMM 2 reads them).  gu_save (both
 * calls that take it): NULL, or the fp32 GEMM-1 accumulators g|u kept for
 * moe_expert_ffn_backward_mx, in moe_expert_ffn's gu_save layout
 * (ceil(max_rows/32)*32 x 2I floats). */
moe_status moe_expert_gemm1_mx(const uint8_t *x_perm_q, const uint8_t *x_perm_sf,
                               const int32_t *offsets, int G, int max_rows, const uint8_t *W13_q,
                               const uint8_t *W13_sf, int d, int I, float clamp, float *gu_save,
                               uint8_t *h_q, uint8_t *h_sf, void *stream);
moe_status moe_expert_gemm2_mx(const uint8_t *h_q, const uint8_t *h_sf, const int32_t *offsets,
                               int G, int max_rows, const uint8_t *W2_q, const uint8_t *W2_sf,
                               const float *row_weight, int S, int d, int I, uint16_t *y_perm,
                               void *stream);

/* MX quantisation along the rows of a stack of matrices, written transposed:
 * src [G, R, C] bf16; output row g*C + c is column c of matrix g (R values)
 * quantised in blocks of 32 along R: q [G*C, R], sf [G*C, moe_mx_sf_pitch(R)].
 * The backward's weight copies: W2 [G, d, I] -> W2^T [G*I, d] quantised along
 * d, W13 [G, 2I, d] -> W13^T [G*d, 2I] quantised along 2I.  Needs R % 32 == 0,
 * G, C >= 1; 16-byte aligned arrays. */
moe_status moe_mx_quantize_t(const uint16_t *src, int G, int R, int C, uint8_t *q, uint8_t *sf,
                             void *stream);

/* Both quantisations of a stack of matrices in one pass over src [G, R, C]
 * bf16: q [G*R, C] / sf [G*R, moe_mx_sf_pitch(C)] along the rows (as
 * moe_mx_quantize of src viewed as [G*R, C]) and qt [G*C, R] / sft [G*C,
 * moe_mx_sf_pitch(R)] along the columns (as moe_mx_quantize_t) -- the
 * forward's and the backward's copies of a weight after each update, for
 * half the HBM reads of the two calls.  Needs R % 128 == 0 and C % 128 == 0
 * (else MOE_ERR_UNSUPPORTED), G >= 1, 16-byte aligned arrays. */
moe_status moe_mx_quantize_both(const uint16_t *src, int G, int R, int C, uint8_t *q,
                                uint8_t *sf, uint8_t *qt, uint8_t *sft, void *stream);

/* Backward of moe_expert_ffn_mx on its rows, in the MX training form: each
 * matmul takes its two operands quantised along its own contraction.
 *   dA[r]   = dY~[r] (W2^T)~[g]^T     dY along d, W2 along d  (fp32 sums)
 *   dw_rows[r] = <h~[r], dA[r]>       h~ the forward's MX h   (r < S)
 *   dH = w dA;  [dg|du][r] = clamped-SwiGLU backward as in moe_backward, from
 *                                     the forward's fp32 g|u
 *   dX_perm[r] = bf16( MX([dg|du][r]) (W13^T)~[g]^T )   along 2I
 *   dW2[g]  = sum_r MXr(dY_perm)[r]^T MXr(bf16(w h~))[r]
 *   dW13[g] = sum_r MXr(bf16([dg|du]))[r]^T MXr(x_perm)[r]
 * MXr: quantised along the group's rows, in blocks of 32 rows from the
 * group's first row (the last block zero-padded), every column of a block one
 * MX block; w h~ and [dg|du] are stored in bf16 first (fp32 sums).
 * gu_save = NULL recomputes g|u and h~ with MX GEMM 1 into the workspace
 * (then x_perm_q/sf and W13_q/sf are read, h_q/h_sf are not); otherwise the
 * forward's gu_save and h_q/h_sf are read.  Needs d % 256 == 0 and
 * I % 128 == 0 (else MOE_ERR_UNSUPPORTED).  Workspace:
 * moe_expert_bwd_mx_workspace_size(G, max_rows, d, I, gu_save == NULL). */
typedef struct {
    int G, max_rows, S, d, I;
    float clamp;
    const int32_t *offsets;       /* [G+1] */
    const uint16_t *x_perm;       /* [R,d] bf16 rows of the forward (dW13) */
    const uint8_t *x_perm_q;      /* [R,d] their MX codes (recompute only) */
    const uint8_t *x_perm_sf;     /* [R,pitch(d)] */
    const uint8_t *W13_q;         /* [G*2I,d] forward W13~ (recompute only) */
    const uint8_t *W13_sf;
    const float *gu_save;         /* forward's g|u, or NULL: recompute */
    const uint8_t *h_q;           /* [R,I] forward's h~ (with gu_save) */
    const uint8_t *h_sf;          /* [R,pitch(I)] */
    const uint8_t *W2t_q;         /* [G*I,d] W2 along d (moe_mx_quantize_t) */
    const uint8_t *W2t_sf;        /* [G*I,pitch(d)] */
    const uint8_t *W13t_q;        /* [G*d,2I] W13 along 2I (moe_mx_quantize_t) */
    const uint8_t *W13t_sf;       /* [G*d,pitch(2I)] */
    const float *row_weight;      /* [S] or NULL (weight 1) */
    const uint16_t *dY_perm;      /* [R,d] bf16 gradient at the rows' outputs */
    const uint8_t *dY_perm_q;     /* [R,d] the same rows MX along d */
    const uint8_t *dY_perm_sf;    /* [R,pitch(d)] */
    uint16_t *dX_perm;            /* [R,d] bf16 out */
    float *dw_rows;               /* [S] out or NULL */
    float *dW13;                  /* [G,2I,d] fp32 out */
    float *dW2;                   /* [G,d,I] fp32 out */
    void *ws;
    size_t ws_bytes;
} moe_expert_bwd_mx_args;
size_t moe_expert_bwd_mx_workspace_size(int G, int max_rows, int d, int I, int recompute);
moe_status moe_expert_ffn_backward_mx(const moe_expert_bwd_mx_args *args, void *stream);

/* Backward of the whole layer with the MX expert matmuls: moe_backward with
 * the expert part of moe_expert_ffn_backward_mx (dY gathered into MX rows
 * for dgrad 2; dW2's operand reads dY's rows through row_token) and the same
 * routing and combine chain.  The bf16 x_perm (dW13, dW_g) is gathered from
 * x; the stages and their events are those of moe_backward.  Workspace:
 * moe_backward_mx_workspace_size(T, d, E, k, I, gu_save == NULL). */
typedef struct {
    int T, d, E, k, I;
    float scaling, clamp;
    const uint16_t *x;            /* [T,d] */
    const uint16_t *W_g;          /* [E,d] */
    const uint8_t *W13_q;         /* forward W13~ [(E+1)*2I,d] (recompute only) */
    const uint8_t *W13_sf;
    const uint8_t *W2t_q;         /* [(E+1)*I,d] */
    const uint8_t *W2t_sf;
    const uint8_t *W13t_q;        /* [(E+1)*d,2I] */
    const uint8_t *W13t_sf;
    const int32_t *ids;           /* [T,k] */
    const float *weights;         /* [T,k] */
    const float *scores_sel;      /* [T,k] */
    const float *row_weight;      /* [S] */
    const int32_t *offsets;       /* [E+2] */
    const int32_t *row_token;     /* [S+T] */
    const int32_t *slot_row;      /* [S] */
    const uint8_t *x_perm_q;      /* [S+T,d] (moe_mx_gather; recompute only) */
    const uint8_t *x_perm_sf;
    const float *gu_save;         /* forward's g|u or NULL: recompute */
    const uint8_t *h_q;           /* forward's h~ (with gu_save) */
    const uint8_t *h_sf;
    const uint16_t *dY;           /* [T,d] */
    uint16_t *dX;                 /* [T,d] bf16 out */
    float *dW_g;                  /* [E,d] */
    float *dW13;                  /* [E+1,2I,d] */
    float *dW2;                   /* [E+1,d,I] */
    float *dlogits;               /* [T,E] or NULL */
    float *dweights;              /* [T,k] or NULL */
    void *ws;
    size_t ws_bytes;
    void *const *stage_events;    /* as in moe_bwd_args, or NULL */
} moe_bwd_mx_args;
size_t moe_backward_mx_workspace_size(int T, int d, int E, int k, int I, int recompute);
moe_status moe_backward_mx(const moe_bwd_mx_args *args, void *stream);

/* Text of a status code (static storage). */
const char *moe_status_string(moe_status s);

/* Synchronises `stream`, returns the device status word of the current
 * device (MOE_OK if no kernel recorded an error since the last call) and
 * resets it. */
moe_status moe_last_device_status(void *stream);

/* Test hook for the bounded wait of moe_expert_ffn_fused: the same call
 * (gu_save = NULL), except that the expert GEMM-2 tiles of the 128-row tile
 * `stall_row_tile` (counted over the groups' row tiles in order) wait for one
 * more GEMM-1 release than will ever come.  Their waits give up after
 * `limit_cycles` SM clock cycles, record MOE_ERR_TIMEOUT in the device status
 * word, and their CTAs drain their copies and MMAs, free their tensor memory
 * and return; the other tiles finish normally.  Nothing traps or hangs, and
 * the context stays usable.  limit_cycles must be in (0, 2^31). */
moe_status moe_selftest_ffn_fused_stall(const uint16_t *x_perm, const int32_t *offsets, int G,
                                        int max_rows, const uint16_t *W13, const uint16_t *W2,
                                        const float *row_weight, int S, int d, int I, float clamp,
                                        uint16_t *h_perm, uint16_t *y_perm, void *ws,
                                        size_t ws_bytes, int stall_row_tile,
                                        long long limit_cycles, void *stream);

/* Tuning: which grouped matmuls may run as 2-SM pairs (two CTAs on two SMs
 * sharing one tcgen05 MMA of 256 rows, each CTA loading half of the weight
 * tile).  `mask` is an OR of the MOE_PAIR_* bits; a paired matmul is used only
 * where the shape suits it (256-wide tiles; for the row-grouped matmuls, on
 * average at least 1024 rows per group).  Results are those of the
 * single-SM form up to the order of fp32 additions inside the tensor core.
 * Process-wide; takes effect at the next call.  Returns the previous mask. */
#define MOE_PAIR_EXPERT_GEMM1 (1 << 1)
#define MOE_PAIR_EXPERT_GEMM2 (1 << 2)
#define MOE_PAIR_DGRAD2 (1 << 3)        /* backward of expert GEMM 2 (+ SwiGLU backward) */
#define MOE_PAIR_DGRAD1 (1 << 4)        /* backward of expert GEMM 1 w.r.t. its input */
#define MOE_PAIR_WGRAD (1 << 5)         /* both weight-gradient matmuls */
int moe_set_gemm_pairs(int mask);

/* Test hook for the bounded waits: launches one block whose mbarrier wait
 * can never complete, with a limit of `limit_cycles` SM clock cycles; the
 * kernel gives up, records MOE_ERR_TIMEOUT in the device status word and
 * returns.  Nothing traps or hangs.  limit_cycles must be in (0, 2^31). */
moe_status moe_selftest_wait_timeout(long long limit_cycles, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */

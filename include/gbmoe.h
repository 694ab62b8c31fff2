/*
 * gbmoe.h -- C ABI of the GB300 (sm_103a) fused mixture-of-experts layer.
 *
 * The layer follows the modular decomposition of
 * "vllm/model_executor/layers/fused_moe/modular_kernel.py" (vllm-cpu
 * 0.11.0.post2 diff view), module comment:
 *     [Router] -> [Quantize-Prepare] -> [Permute-Experts-Unpermute] -> [Finalize]
 * with its problem statement from _moe_problem_size: E experts, M tokens,
 * hidden size K, intermediate size N, topk experts per token,
 * w1 (E, 2N, K) and w2 (E, K, N); and its two activation formats from
 * FusedMoEActivationFormat: Standard (M, K) and BatchedExperts
 * (E, max_tokens, K).  The batched format is masked by a device-resident
 * per-expert token count, as in "EP: CUDA-graph-safe HT internode
 * dispatch+combine (worst-tokens mode)" (uccl pull request 7), so that the
 * whole layer can be captured in a CUDA graph without reading counts on the
 * host.
 *
 * Conventions for every call below:
 *   - Pointers are DEVICE pointers to caller-owned memory unless stated
 *     otherwise; every tensor is row-major with its last index contiguous.
 *     bf16 is IEEE bfloat16 bits (uint16), e4m3 is the OCP "E4M3FN" byte.
 *   - The library allocates no device memory and never synchronises the
 *     host: each call validates its arguments, enqueues kernels on `stream`
 *     and returns.  Scratch memory comes from a caller buffer `ws` of at least
 *     moe_workspace_size(...) bytes, 256-byte aligned.
 *   - Tensors read by the tensor-core GEMMs (x / A rows, w1, w2, H) must start
 *     on a 16-byte boundary.
 *   - Return value: GBMOE_OK, or GBMOE_INVALID_ARG (null pointer, bad size,
 *     K or N not a multiple of 128, topk > E, workspace too small,
 *     misaligned pointer), GBMOE_UNSUPPORTED (dtype, or a device that is not
 *     sm_103), GBMOE_CUDA_ERROR (a launch failed; see gbmoe_last_cuda_error).
 *     Nothing is enqueued when a call returns GBMOE_INVALID_ARG or
 *     GBMOE_UNSUPPORTED (arguments are checked before the first launch); a
 *     call of several launches that returns GBMOE_CUDA_ERROR may have
 *     enqueued the launches before the failing one.
 *   - Errors in the DATA (an expert id outside [0, E), a batched count
 *     outside [0, T], a device wait that ran out of time) cannot be seen on
 *     the host without a sync.  Kernels skip the offending element and OR a
 *     GBMOE_ERR_* bit into the caller's device word `err_word` (may be NULL
 *     where noted); read it after synchronising.  No kernel traps.
 *   - M == 0 (or E * T == 0) is a valid no-op and returns GBMOE_OK.
 *   - `stream` must belong to the device that is current on the calling
 *     thread (cudaSetDevice); calls that keep per-device state refuse a
 *     stream of another device with GBMOE_INVALID_ARG.
 */
#ifndef GBMOE_H
#define GBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gbmoe_stream_t; /* a cudaStream_t; NULL = legacy default stream */
typedef struct CUevent_st *gbmoe_event_t;   /* a cudaEvent_t */

typedef enum {
    GBMOE_OK = 0,
    GBMOE_INVALID_ARG = 1,
    GBMOE_UNSUPPORTED = 2,
    GBMOE_CUDA_ERROR = 3
} gbmoe_status_t;

/* element type of activations / weights fed to the expert GEMMs:
 * GBMOE_FP8_E4M3          e4m3 with fp32 block scales: 1 x 128 groups of a
 *                         token's activations, 128 x 128 blocks of weights
 *                         (K and N at most 16384 for the GEMMs);
 * GBMOE_FP8_E4M3_CHANNEL  e4m3 with one fp32 scale per token of the
 *                         activations and one per output channel (row) of
 *                         w1 and w2 -- the quant config's
 *                         per_act_token_quant and per_out_ch_quant
 *                         (FusedMoEPermuteExpertsUnpermute's quant
 *                         properties); the scale rule is that of
 *                         moe_quant_fp8_group with a group as wide as the
 *                         row;
 * GBMOE_FP8_E4M3_TENSOR   e4m3 with one fp32 scale for a whole activation
 *                         tensor (the layer's input; H) -- per_act_token_quant
 *                         off, no block shape -- and per-channel weight
 *                         scales as above (per-tensor weight scales are
 *                         per-channel scales of equal value). */
enum { GBMOE_BF16 = 0, GBMOE_FP8_E4M3 = 1, GBMOE_FP8_E4M3_CHANNEL = 2,
       GBMOE_FP8_E4M3_TENSOR = 3 };
/* router score function */
enum { GBMOE_SOFTMAX = 0, GBMOE_SIGMOID = 1 };
/* gated activation of the experts (FusedMoEPermuteExpertsUnpermute.activation):
 * "silu" -> silu_and_mul, h = silu(g) * u with silu(z) = z / (1 + exp(-z));
 * "gelu" -> gelu_and_mul, h = gelu(g) * u with the exact
 * gelu(z) = z / 2 * (1 + erf(z / sqrt 2)) */
enum { GBMOE_ACT_SILU = 0, GBMOE_ACT_GELU = 1 };
/* which call a workspace is sized for (moe_workspace_size) */
enum {
    GBMOE_WS_ALIGN = 0,    /* moe_align_permute                       */
    GBMOE_WS_BATCHED = 2,  /* moe_batched_masked_experts              */
    GBMOE_WS_FORWARD = 3,  /* moe_forward (the whole Standard layer)  */
    GBMOE_WS_SHARED = 4,   /* moe_shared_expert_forward (N = shared intermediate size;
                              dtype GBMOE_BF16, GBMOE_FP8_E4M3 or
                              GBMOE_FP8_E4M3_CHANNEL) */
    GBMOE_WS_EP_DISPATCH = 6  /* moe_ep_dispatch: M_or_T = M tokens per shard, E = all
                                 routed experts, N = the number of shards G  */
};

/* bits OR-ed into *err_word by the kernels */
#define GBMOE_ERR_BAD_EXPERT_ID 0x1  /* an id outside [0, E): the pair is skipped  */
#define GBMOE_ERR_COUNT_RANGE 0x2    /* a batched count outside [0, T]: clamped    */
#define GBMOE_ERR_TIMEOUT 0x4        /* a pipeline wait ran out of time: tile left  */

/* Status code as a short English string (static storage). */
const char *gbmoe_status_string(gbmoe_status_t status);

/* The cudaError_t (as int) of the last failed launch in this process, 0 if none. */
int gbmoe_last_cuda_error(void);

/* Bytes of workspace a call needs.  `which` is a GBMOE_WS_* value; M_or_T is
 * M for the Standard calls and T (max tokens per expert) for the batched one.
 * E is the number of local experts (the first dimension of w1 / w2).
 * Returns 0 for invalid arguments. */
size_t moe_workspace_size(int which, int M_or_T, int E, int N, int K, int topk,
                          int dtype);

/* [Router] -- the first stage of the module comment of modular_kernel.py;
 * FusedMoEModularKernel.forward receives its topk_weights / topk_ids.
 * Per token t:
 *   score_fn GBMOE_SOFTMAX: the topk largest logits (softmax is monotone);
 *     weight = softmax(logits[t])[e], divided by its sum over the chosen
 *     experts when renormalize != 0.
 *   score_fn GBMOE_SIGMOID: s_e = sigmoid(v_e), v_e = logits[t,e] + bias[e]
 *     (fp32 add).  The E experts form n_groups contiguous groups; a group's
 *     key is the fp32 sum of the scores of its two largest v, each score the
 *     fp32 rounding of an fp64 sigmoid; the topk_groups groups with the
 *     largest keys are kept, and the topk experts with the largest v (the
 *     sigmoid's order) among them are chosen; weight = s_e, renormalised as
 *     above.  n_groups <= 1 means no group limit.
 *   Ties go to the lower expert (group) index; a row lists its experts in
 *   descending score order.
 * logits (M, E) fp32; bias (E) fp32 or NULL (sigmoid only);
 * topk_ids (M, topk) int32 out; topk_weights (M, topk) fp32 out.
 * 1 <= topk <= E <= 512; for sigmoid, E % n_groups == 0 and
 * topk <= topk_groups * (E / n_groups).  err_word unused (may be NULL). */
gbmoe_status_t moe_topk_route(const float *logits, const float *bias, int M,
                              int E, int topk, int score_fn, int n_groups,
                              int topk_groups, int renormalize,
                              int32_t *topk_ids, float *topk_weights,
                              int32_t *err_word, gbmoe_stream_t stream);

/* Expert ids and the expert-parallel map.  The router picks among E_global
 * (routed, global) experts; this shard holds the E local experts of w1 / w2.
 * expert_map (E_global) int32, as the expert_map argument of
 * FusedMoEModularKernel.forward: expert_map[g] is the local id of global
 * expert g, or -1 when g is not on this shard -- its (token, slot) pairs are
 * not computed here and add nothing to the output.  expert_map NULL: ids are
 * local already and E_global must equal E.  A routed id outside
 * [0, E_global), or mapped outside [-1, E), is invalid: it is skipped and
 * sets GBMOE_ERR_BAD_EXPERT_ID. */

/* count_expert_num_tokens as named in modular_kernel.py
 * (FusedMoEModularKernel._maybe_chunk_fused_experts) and the
 * ExpertTokensMetadata.expert_num_tokens it fills:
 * counts[l] = #{p < M*topk : topk_ids[p] maps to local expert l}, computed on
 * the device.  topk_ids (M, topk) int32; counts (E) int32 out (overwritten). */
gbmoe_status_t moe_count_expert_tokens(const int32_t *topk_ids, int M,
                                       int topk, int E_global,
                                       const int32_t *expert_map, int E,
                                       int32_t *counts, int32_t *err_word,
                                       gbmoe_stream_t stream);

/* The "Permute" of [Permute-Experts-Unpermute]: a stable counting sort of the
 * P = M*topk (token, slot) pairs by local expert.  Pair p = t*topk + j.
 *   counts (E) int32 out, or NULL: counts[l] as in moe_count_expert_tokens,
 *     the ExpertTokensMetadata.expert_num_tokens of the pages;
 *   offsets (E+1) int32 out: offsets[0] = 0, offsets[l+1] = offsets[l] + counts[l];
 *   sorted_pair_ids (M*topk) int32 out: sorted_pair_ids[offsets[l] + r] is the
 *     r-th pair, in ascending p, routed to local expert l (entries at and
 *     beyond offsets[E] are left unwritten);
 *   inv (M*topk) int32 out: inv[p] = the position of p in sorted_pair_ids,
 *     -1 for a pair that is not computed here (invalid id, or an expert that
 *     is not local).
 * ws: moe_workspace_size(GBMOE_WS_ALIGN, M, E, 0, 0, topk, 0) bytes (one
 * histogram per chunk of 2048 pairs).  err_word may be NULL. */
gbmoe_status_t moe_align_permute(const int32_t *topk_ids, int M, int topk,
                                 int E_global, const int32_t *expert_map, int E,
                                 int32_t *counts, int32_t *offsets,
                                 int32_t *sorted_pair_ids, int32_t *inv,
                                 void *ws, size_t ws_bytes, int32_t *err_word,
                                 gbmoe_stream_t stream);

/* [Quantize-Prepare] (FusedMoEPrepareAndFinalize.prepare quantises the
 * activations before the experts run), per-token-group FP8:
 * for each token t and each group g of `group` consecutive columns, with
 * v[t,k] = x[t,k] * row_weights[t] (an fp32 product; v = x when row_weights
 * is NULL -- the weights are given with apply_router_weight_on_input, when
 * prepare applies the router weight to the activations):
 *   s = max(max_k |v[t,k]|, 1e-12) / 448   (fp32, IEEE division)
 *   q[t,k] = e4m3(v[t,k] / s)               (round to nearest even, saturating at 448)
 * x (M, K) bf16; row_weights (M) fp32 or NULL; q (M, K) e4m3 out;
 * scales (M, K/group) fp32 out.  group must be 128 or K (one group per row:
 * the per-token scales of GBMOE_FP8_E4M3_CHANNEL, and with x = a weight
 * tensor viewed as (E*R, C), its per-channel scales); K % 128 == 0. */
gbmoe_status_t moe_quant_fp8_group(const uint16_t *x, const float *row_weights,
                                   int M, int K, int group, uint8_t *q,
                                   float *scales, gbmoe_stream_t stream);

/* The quantiser with one group holding a whole tensor (dynamic per-tensor
 * scale): over rows t < n (n = *n_rows when n_rows is given, a device
 * int32 -- the row count a previous kernel wrote, e.g. offsets[E] -- else M),
 * with v[t,k] = x[t,k] * row_weights[t] as above,
 *   s = max(max_{t<n,k} |v[t,k]|, 1e-12) / 448,  q[t,k] = e4m3(v[t,k] / s),
 * and row_scales[t] = s for every t < n, so that the permute and GEMM calls
 * take the tensor's scale as a per-row one (dtype GBMOE_FP8_E4M3_TENSOR).
 * Rows t >= n are left unwritten.  amax_ws: 4 bytes of caller device
 * memory, overwritten (the maximum is reduced there; max is order-free, so
 * the result is deterministic).  Three launches on `stream` (a 4-byte
 * clear, the maximum, the codes).  K % 128 == 0; x, q 16-byte aligned. */
gbmoe_status_t moe_quant_fp8_tensor(const uint16_t *x, const float *row_weights,
                                    int M, int K, const int32_t *n_rows,
                                    uint8_t *q, float *row_scales,
                                    uint32_t *amax_ws, gbmoe_stream_t stream);

/* The same quantiser with a static per-tensor scale (the quant config's
 * a1_scale / a2_scale): scale is a DEVICE fp32 scalar (4-byte aligned), and
 *   q[t,k] = e4m3(v[t,k] / scale)   (IEEE division, saturating at +-448),
 *   row_scales[t] = scale            for every t < n,
 * with v, n_rows, x, q, row_scales as in moe_quant_fp8_tensor.  One launch
 * on `stream`.  K % 128 == 0; x, q 16-byte aligned. */
gbmoe_status_t moe_quant_fp8_tensor_static(const uint16_t *x, const float *row_weights,
                                           int M, int K, const int32_t *n_rows,
                                           const float *scale, uint8_t *q, float *row_scales,
                                           gbmoe_stream_t stream);

/* The same quantiser over block x block tiles of a weight matrix, for
 * preparing FP8 expert weights (not part of the timed layer):
 * w (R, C) bf16 -> q (R, C) e4m3 and scales (R/block, C/block) fp32, one
 * scale per tile from the tile's largest magnitude.  block must be 128,
 * R % 128 == 0 and C % 128 == 0.  w1 (E, 2N, K) is passed as R = E*2N,
 * C = K; w2 (E, K, N) as R = E*K, C = N. */
gbmoe_status_t moe_quant_fp8_block(const uint16_t *w, int64_t R, int C,
                                   int block, uint8_t *q, float *scales,
                                   gbmoe_stream_t stream);

/* The data movement of the "Permute": the rows of the first GEMM in sorted
 * order, A[i] = x[sorted_pair_ids[i] / topk] for i < offsets[E] (rows at and
 * beyond offsets[E] are left unwritten).
 * dtype GBMOE_BF16: x (M, K) bf16 -> A (M*topk, K) bf16; scales unused;
 *   row_weights (M*topk) fp32 or NULL: with apply_router_weight_on_input,
 *   A[i] = bf16(x[t] * row_weights[p]) with p = sorted_pair_ids[i].
 * dtype GBMOE_FP8_E4M3: x (M, K) e4m3 with x_scales (M, K/128) fp32 ->
 *   A (M*topk, K) e4m3 with A_scales stored GROUP-MAJOR: A_scales[g * ld + i]
 *   is the scale of row i, K block g, with ld = M*topk rounded up to a
 *   multiple of 4 (a (K/128, ld) array), so that the scales of one K block
 *   of consecutive rows are contiguous for the GEMM's TMA loads.
 *   row_weights must be NULL (the FP8 rows take the weight in
 *   moe_quant_fp8_group, before the codes are chosen).
 * dtype GBMOE_FP8_E4M3_CHANNEL or GBMOE_FP8_E4M3_TENSOR: x (M, K) e4m3 with
 *   x_scales (M) fp32 -> A (M*topk, K) e4m3 with A_scales (M*topk) fp32, one
 *   per row; row_weights must be NULL.
 * K % 128 == 0; x and A 16-byte aligned. */
gbmoe_status_t moe_permute_rows(const void *x, const float *x_scales,
                                const float *row_weights,
                                const int32_t *sorted_pair_ids,
                                const int32_t *offsets, int M, int topk, int E,
                                int K, int dtype, void *A, float *A_scales,
                                gbmoe_stream_t stream);

/* moe_quant_fp8_group (group 128) and moe_permute_rows (dtype
 * GBMOE_FP8_E4M3) in one pass: each token's 1 x 128 groups are quantised
 * once and their codes and scales written straight to the permuted rows of
 * the token's pairs, A[inv[p]] for p = t*topk + j (pairs with inv[p] < 0,
 * not routed to a local expert, are skipped).  The results equal the two
 * calls' bit for bit.
 * x (M, K) bf16; row_weights (M) fp32 or NULL (apply_router_weight_on_input,
 * topk 1: the fp32 product of a row and its weight is quantised); inv
 * (M*topk) int32 from moe_align_permute; A (M*topk, K) e4m3 and A_scales
 * group-major (K/128, ld), ld = M*topk rounded up to 4, as
 * moe_permute_rows writes them.  K % 128 == 0; x and A 16-byte aligned. */
gbmoe_status_t moe_quant_fp8_group_permute(const uint16_t *x,
                                           const float *row_weights, int M,
                                           int K, const int32_t *inv, int topk,
                                           uint8_t *A, float *A_scales,
                                           gbmoe_stream_t stream);

/* The same for one scale per token (moe_quant_fp8_group with group = K, and
 * moe_permute_rows with dtype GBMOE_FP8_E4M3_CHANNEL) in one pass: a row's
 * codes and its scale go to every permuted row of the token's pairs,
 * A[inv[p]] and A_scales[inv[p]] (pairs with inv[p] < 0 skipped); equal to
 * the two calls bit for bit.  Arguments as moe_quant_fp8_group_permute, with
 * A_scales (M*topk) fp32 (4-byte aligned). */
gbmoe_status_t moe_quant_fp8_row_permute(const uint16_t *x,
                                         const float *row_weights, int M,
                                         int K, const int32_t *inv, int topk,
                                         uint8_t *A, float *A_scales,
                                         gbmoe_stream_t stream);

/* The same for one scale for the whole of x (dtype GBMOE_FP8_E4M3_TENSOR):
 * the scale is scale[0] (a DEVICE fp32, static) or, when scale is NULL, the
 * maximum over all M rows / 448 (reduced in amax_ws, 4 bytes of caller
 * device memory, overwritten); every token's codes and the scale go to the
 * permuted rows of its pairs, A[inv[p]] and A_scales[inv[p]], as
 * moe_quant_fp8_tensor(_static) followed by moe_permute_rows would write
 * them, bit for bit.  Arguments otherwise as moe_quant_fp8_row_permute;
 * three launches with a dynamic scale, one with a static one. */
gbmoe_status_t moe_quant_fp8_tensor_permute(const uint16_t *x,
                                            const float *row_weights, int M,
                                            int K, const int32_t *inv, int topk,
                                            const float *scale, uint8_t *A,
                                            float *A_scales, uint32_t *amax_ws,
                                            gbmoe_stream_t stream);

/* First expert GEMM with the gated activation fused into its epilogue:
 * the first GEMM of FusedMoEPermuteExpertsUnpermute.apply followed by its
 * gated activation (and, for block-scaled e4m3, the requantisation of the
 * result), with activation "silu" (silu_and_mul: the output is half as wide
 * as the GEMM).  For every sorted position i in [offsets[e], offsets[e+1]):
 *   g[n] = A[i] . w1[e, n, :],   u[n] = A[i] . w1[e, N + n, :]   (n < N)
 *   H[i, n] = silu(g[n]) * u[n],  silu(z) = z / (1 + exp(-z))
 * Rows [0, N) of w1[e] are the gate, rows [N, 2N) the up projection.
 * A (M*topk, K) is in sorted order (moe_permute_rows); rows of H at and beyond
 * offsets[E] are left unwritten.
 * dtype GBMOE_BF16: A bf16, w1 (E, 2N, K) bf16, H (M*topk, N) bf16;
 *   A_scales / w1_scales / H_scales unused (NULL).
 * dtype GBMOE_FP8_E4M3: A e4m3 with group-major A_scales (K/128, ld) fp32
 *   (moe_permute_rows; ld = M*topk rounded up to 4, 16-byte aligned); w1
 *   e4m3 with w1_scales (E, 2N/128, K/128) fp32 (128 x 128 blocks); each
 *   128-wide K block is accumulated in fp32 and scaled by A_scale * w1_scale
 *   before it is added.  H is written as e4m3 with group-major H_scales
 *   (N/128, ld) fp32, requantised per 128-group of a row with the
 *   moe_quant_fp8_group rule.
 * dtype GBMOE_FP8_E4M3_CHANNEL or GBMOE_FP8_E4M3_TENSOR: A e4m3 with
 *   A_scales (M*topk) fp32, w1 e4m3 with w1_scales (E, 2N) fp32; the whole K
 *   is accumulated in fp32 and scaled once,
 *   g[n] = A_scale[i] * w1_scale[e, n] * (codes dot product).
 *   H (M*topk, N) is written in bf16 (H_scales unused): its scale spans at
 *   least a whole row, so the caller quantises H with moe_quant_fp8_group
 *   (group = N; CHANNEL) or moe_quant_fp8_tensor (n_rows = offsets + E;
 *   TENSOR) before moe_grouped_gemm_down.
 * Accumulation is fp32.  N % 128 == 0, K % 128 == 0.  err_word may be NULL. */
gbmoe_status_t moe_grouped_gemm_gate_up_silu(
    const void *A, const float *A_scales, const int32_t *offsets, int M,
    int topk, int E, int N, int K, const void *w1, const float *w1_scales,
    int dtype, void *H, float *H_scales, int32_t *err_word,
    gbmoe_stream_t stream);

/* The same GEMM with activation "gelu" (gelu_and_mul):
 * H[i, n] = gelu(g[n]) * u[n], gelu the exact erf form above. */
gbmoe_status_t moe_grouped_gemm_gate_up_gelu(
    const void *A, const float *A_scales, const int32_t *offsets, int M,
    int topk, int E, int N, int K, const void *w1, const float *w1_scales,
    int dtype, void *H, float *H_scales, int32_t *err_word,
    gbmoe_stream_t stream);

/* Second expert GEMM with the router weight fused into its epilogue
 * (the experts own the weight application, which
 * FusedMoEPermuteExpertsUnpermute.finalize_weight_and_reduce_impl hands to
 * [Finalize]).  For every sorted position i of expert e, with
 * p = sorted_pair_ids[i]:
 *   y_slot[p, k] = topk_weights[p] * (H[i, :] . w2[e, k, :])      (k < K)
 * y_slot (M, topk, K) bf16 is the fused_expert_output of
 * FusedMoEPrepareAndFinalize.finalize, already weighted; its rows of pairs
 * that are not computed here are not written.  topk_weights NULL: no weight
 * (apply_router_weight_on_input applied it to the input instead).
 * dtype GBMOE_BF16: H (M*topk, N) bf16, w2 (E, K, N) bf16.
 * dtype GBMOE_FP8_E4M3: H e4m3 + group-major H_scales (N/128, ld), ld =
 *   M*topk rounded up to 4 (as written by the gate/up call); w2 e4m3 +
 *   w2_scales (E, K/128, N/128).
 * dtype GBMOE_FP8_E4M3_CHANNEL or GBMOE_FP8_E4M3_TENSOR: H e4m3 + H_scales
 *   (M*topk) fp32, one per row; w2 e4m3 + w2_scales (E, K) fp32, one per
 *   output channel.
 * Accumulation fp32.  err_word may be NULL. */
gbmoe_status_t moe_grouped_gemm_down(
    const void *H, const float *H_scales, const int32_t *sorted_pair_ids,
    const int32_t *offsets, const float *topk_weights, int M, int topk, int E,
    int N, int K, const void *w2, const float *w2_scales, int dtype,
    uint16_t *y_slot, int32_t *err_word, gbmoe_stream_t stream);

/* [Finalize]: TopKWeightAndReduce.apply and FusedMoEPrepareAndFinalize.finalize
 * (output (M, K) from fused_expert_output (M, topk, K)).  The weights are
 * already applied, so
 *   out[t, k] = bf16( sum_{j = 0 .. topk-1} y_slot[t, j, k] )
 * summed in fp32 in slot order j = 0, 1, ... (deterministic), skipping the
 * pairs with inv[t*topk + j] < 0 when inv is not NULL.
 * y_slot (M, topk, K) bf16; out (M, K) bf16. */
gbmoe_status_t moe_unpermute_weighted_reduce(const uint16_t *y_slot,
                                             const int32_t *inv, int M,
                                             int topk, int K, uint16_t *out,
                                             gbmoe_stream_t stream);

/* Both expert GEMMs in the BatchedExperts format (E, T, K), masked by the
 * device-resident expert_num_tokens as the masked grouped GEMM of the
 * worst-tokens mode reads it: for every expert e and row r < c_e,
 * c_e = min(max(expert_num_tokens[e], 0), T),
 *   h = silu(x_b[e,r] . w1[e, 0:N]^T) * (x_b[e,r] . w1[e, N:2N]^T)
 *   y_b[e, r, :] = h . w2[e]^T           (unweighted; no reduction)
 * (gelu in place of silu when activation is GBMOE_ACT_GELU).
 * Rows r >= c_e of x_b are never read and rows r >= c_e of y_b are never
 * written.  A count outside [0, T] is clamped and sets GBMOE_ERR_COUNT_RANGE.
 * No count is read on the host, so the call can be captured in a CUDA graph
 * and replayed with new counts.
 * dtype GBMOE_BF16: x_b (E, T, K) bf16, w1 (E, 2N, K), w2 (E, K, N) bf16;
 *   x_b_scales, w1_scales, w2_scales ignored.
 * dtype GBMOE_FP8_E4M3 (the experts' side of the prepare step's per-token-
 *   group quantisation): x_b (E, T, K) e4m3 codes with x_b_scales
 *   (E*T, K/128) fp32 row-major, one scale per row and 128-group (the layout
 *   moe_quant_fp8_group writes for x_b viewed as (E*T, K)); w1/w2 e4m3 with
 *   their 128 x 128 block scales w1_scales (E, 2N/128, K/128) and
 *   w2_scales (E, K/128, N/128).  The products are promoted per 128-wide K
 *   block, h is requantised to e4m3 per row and 128-group inside ws, and the
 *   down projection reads it back with those scales.  Scales of padded rows
 *   are never used.  The other e4m3 dtypes return GBMOE_UNSUPPORTED.
 * y_b (E, T, K) bf16 in both cases.
 * ws: moe_workspace_size(GBMOE_WS_BATCHED, T, E, N, K, 1, dtype) bytes. */
gbmoe_status_t moe_batched_masked_experts(
    const void *x_b, const float *x_b_scales,
    const int32_t *expert_num_tokens, int E, int T, int N, int K,
    const void *w1, const float *w1_scales, const void *w2,
    const float *w2_scales, int dtype, int activation, uint16_t *y_b, void *ws,
    size_t ws_bytes, int32_t *err_word, gbmoe_stream_t stream);

/* The whole layer in the Standard format, FusedMoEModularKernel.forward
 * without shared experts: route -> count -> align/permute -> [quantise] ->
 * gate/up GEMM + SiLU*mul -> down GEMM + weight -> ordered reduce, all on
 * `stream`.
 * x (M, K) bf16; logits (M, E_global) fp32; bias (E_global) fp32 or NULL;
 * expert_map (E_global) or NULL and E local experts, as described above
 * moe_count_expert_tokens (the output then holds the local experts' part);
 * apply_router_weight_on_input != 0 (topk must be 1): the router weight
 * multiplies the activations (before FP8 quantisation) instead of the expert
 * output, out[t] = expert(w[t] * x[t]);
 * activation: GBMOE_ACT_SILU or GBMOE_ACT_GELU;
 * dtype GBMOE_BF16: w1 (E, 2N, K) / w2 (E, K, N) bf16, scales NULL;
 * dtype GBMOE_FP8_E4M3: w1/w2 e4m3 with their block scales; the activations
 *   are quantised per token in groups of 128 and H is requantised.
 * dtype GBMOE_FP8_E4M3_CHANNEL: w1/w2 e4m3 with their per-channel scales
 *   (E, 2N) / (E, K); the activations are quantised with one scale per
 *   token, H is kept in bf16 and quantised per token before the second GEMM.
 * dtype GBMOE_FP8_E4M3_TENSOR: the same weights; x is quantised with one
 *   scale for all M tokens and H with one for all its computed rows.  The
 *   scales are the tensors' own maxima / 448 (dynamic), or the caller's
 *   static scales: a1_scale for x and a2_scale for H (the quant config's
 *   a1_scale / a2_scale, FusedMoEPrepareAndFinalize.prepare), each a DEVICE
 *   fp32 scalar (4-byte aligned) or NULL for the dynamic scale; codes are
 *   e4m3(v / scale), saturating at +-448.  With any other dtype both must be
 *   NULL (GBMOE_INVALID_ARG otherwise).
 * out (M, K) bf16.  topk_ids / topk_weights (M, topk) may be NULL; when given
 * they receive the router's output (global ids).
 * ws: moe_workspace_size(GBMOE_WS_FORWARD, M, E, N, K, topk, dtype) bytes.
 * err_word may be NULL. */
gbmoe_status_t moe_forward(const uint16_t *x, const float *logits,
                           const float *bias, int M, int K, int N, int E_global,
                           const int32_t *expert_map, int E, int topk,
                           int score_fn, int n_groups, int topk_groups,
                           int renormalize, int apply_router_weight_on_input,
                           int activation, int dtype, const void *w1,
                           const float *w1_scales,
                           const void *w2, const float *w2_scales,
                           const float *a1_scale, const float *a2_scale,
                           uint16_t *out, int32_t *topk_ids,
                           float *topk_weights, void *ws, size_t ws_bytes,
                           int32_t *err_word, gbmoe_stream_t stream);

/* moe_forward in chunks of at most chunk_size tokens, one after the other on
 * `stream`, as FusedMoEModularKernel._maybe_chunk_fused_experts does to bound
 * its workspaces -- but with every chunk's counts computed on the device (the
 * pages copy them to the host per chunk), so the whole loop stays
 * capturable.  Each token's result is the same as unchunked, bit for bit --
 * except with GBMOE_FP8_E4M3_TENSOR and dynamic scales, which are then taken
 * per chunk (as the chunk loop quantises each chunk on its own); static
 * scales (a1_scale, a2_scale) give the unchunked result.
 * Arguments as moe_forward (topk_ids / topk_weights may be NULL);
 * ws: moe_workspace_size(GBMOE_WS_FORWARD, min(M, chunk_size), E, N, K,
 * topk, dtype) bytes. */
gbmoe_status_t moe_forward_chunked(const uint16_t *x, const float *logits,
                                   const float *bias, int M, int K, int N,
                                   int E_global, const int32_t *expert_map,
                                   int E, int topk, int score_fn, int n_groups,
                                   int topk_groups, int renormalize,
                                   int apply_router_weight_on_input,
                                   int activation, int dtype, const void *w1,
                                   const float *w1_scales, const void *w2,
                                   const float *w2_scales, const float *a1_scale,
                                   const float *a2_scale, uint16_t *out,
                                   int32_t *topk_ids, float *topk_weights,
                                   int chunk_size, void *ws, size_t ws_bytes,
                                   int32_t *err_word, gbmoe_stream_t stream);

/* The shared experts of the layer: a dense gated MLP applied to every token
 * (the shared_experts of FusedMoEModularKernel.forward, whose output it
 * returns beside the routed one; the SharedExperts page runs them on an
 * auxiliary stream).  For every token t:
 *   h = act(x[t] . w1s[0:Ns]^T) * (x[t] . w1s[Ns:2Ns]^T),
 *   out_shared[t] = h . w2s^T
 * x (M, K) bf16; w1s (2Ns, K), w2s (K, Ns) (the shared experts stacked
 * along Ns); out_shared (M, K) bf16; activation GBMOE_ACT_*.
 * dtype GBMOE_BF16: w1s, w2s bf16, the scale pointers unused (may be NULL).
 * dtype GBMOE_FP8_E4M3: w1s, w2s e4m3 with 128 x 128 block scales
 * w1s_scales (2Ns/128, K/128) and w2s_scales (K/128, Ns/128) fp32 (4-byte
 * aligned; moe_quant_fp8_block makes them); x is quantised inside the call
 * in 1 x 128 groups and h in 1 x 128 groups along Ns, as moe_forward does
 * for the routed experts; K and Ns at most 16384.
 * dtype GBMOE_FP8_E4M3_CHANNEL: w1s, w2s e4m3 with one fp32 scale per row,
 * w1s_scales (2Ns) and w2s_scales (K), 16-byte aligned (moe_quant_fp8_group
 * with a group as wide as the row makes them); x is quantised with one scale
 * per token and h, kept in bf16, with one scale per row, as moe_forward does.
 * Other dtypes: GBMOE_UNSUPPORTED.  Runs the grouped-GEMM kernels with one
 * expert holding all M rows (e4m3: after the group quantisation of x and a
 * transpose of its scales).  ws: moe_workspace_size(GBMOE_WS_SHARED, M, 1,
 * Ns, K, 1, dtype). */
gbmoe_status_t moe_shared_expert_forward(const uint16_t *x, int M, int K, int Ns,
                                         const void *w1s, const float *w1s_scales,
                                         const void *w2s, const float *w2s_scales,
                                         int dtype, int activation, uint16_t *out_shared,
                                         void *ws, size_t ws_bytes, int32_t *err_word,
                                         gbmoe_stream_t stream);

/* moe_forward with the shared experts overlapped on an auxiliary stream
 * (the MULTI_STREAM_OVERLAPPED order of the SharedExperts page): records
 * ev_input_ready on `stream`, makes aux_stream wait for it, enqueues
 * moe_shared_expert_forward on aux_stream and records ev_output_ready
 * there, enqueues the routed layer (moe_forward) on `stream`, and makes
 * `stream` wait for ev_output_ready -- so work enqueued on `stream` after
 * the call sees both out (routed) and out_shared.  The events are created by
 * the caller (cudaEvent_t; timing may be disabled).  aux_stream NULL: both
 * run on `stream` one after the other.  The fork/join is capturable in a
 * CUDA graph when `stream` is being captured.
 * Arguments as moe_forward, plus Ns, w1s, w1s_scales, w2s, w2s_scales and
 * out_shared as moe_shared_expert_forward, whose dtype is shared_dtype
 * (GBMOE_BF16, GBMOE_FP8_E4M3 or GBMOE_FP8_E4M3_CHANNEL, independent of the
 * routed experts' dtype);
 * ws_shared: moe_workspace_size(GBMOE_WS_SHARED, M, 1, Ns, K, 1,
 * shared_dtype) bytes, separate from ws.  Both calls' arguments are checked
 * before anything is enqueued. */
gbmoe_status_t moe_forward_shared(const uint16_t *x, const float *logits,
                                  const float *bias, int M, int K, int N,
                                  int E_global, const int32_t *expert_map,
                                  int E, int topk, int score_fn, int n_groups,
                                  int topk_groups, int renormalize,
                                  int apply_router_weight_on_input,
                                  int activation, int dtype, const void *w1,
                                  const float *w1_scales, const void *w2,
                                  const float *w2_scales, const float *a1_scale,
                                  const float *a2_scale, uint16_t *out,
                                  void *ws, size_t ws_bytes, int Ns,
                                  const void *w1s, const float *w1s_scales,
                                  const void *w2s, const float *w2s_scales,
                                  int shared_dtype, uint16_t *out_shared, void *ws_shared,
                                  size_t ws_shared_bytes, int32_t *err_word,
                                  gbmoe_stream_t stream,
                                  gbmoe_stream_t aux_stream,
                                  gbmoe_event_t ev_input_ready,
                                  gbmoe_event_t ev_output_ready);

/* Expert-parallel dispatch in the worst-tokens mode of "EP: CUDA-graph-safe
 * HT internode dispatch+combine (worst-tokens mode)" (uccl pull request 7 and
 * the vLLM commit message under it), for G shards whose buffers are in this
 * GPU's memory.  Shard r (r < G) holds tokens x[r] (M, K), of which the
 * first num_tokens[r] (a DEVICE int32, clamped to [0, M]) are valid, with
 * their routed expert ids topk_ids[r] (M, topk) int32 in [0, E).  Shard g
 * owns the E / G experts [g*E/G, (g+1)*E/G).  Each valid (token, slot) pair
 * goes to the receive block of its expert:
 *   recv_x (E, worst_tokens, K): recv_x[e, pos] = x[r, t] for the pos-th
 *     pair routed to e, pairs taken in ascending order of (r, t, slot);
 *     the E/G experts of shard g are rows [g*E/G, (g+1)*E/G): that shard's
 *     static worst-case receive buffer, in the BatchedExperts layout;
 *   recv_counts (E) int32, device: rows received per expert (the per-expert
 *     count tensor the masked grouped GEMM reads inside a graph: pass
 *     recv_x + g*(E/G)*worst_tokens*K and recv_counts + g*(E/G) to
 *     moe_batched_masked_experts for shard g);
 *   recv_pos (G, M, topk) int32: pos of each pair, -1 for pairs of padded
 *     tokens and of invalid ids (those are skipped; invalid ids also set
 *     GBMOE_ERR_BAD_EXPERT_ID).
 * worst_tokens is the static per-expert capacity, G * M covers every case
 * (the pages size it as the padded step tokens times the number of
 * dispatchers); pairs beyond it are dropped (pos -1), the count clamped and
 * GBMOE_ERR_COUNT_RANGE set.  Rows of recv_x at and beyond a count are not
 * written.  No count is read on the host and no loop runs over the padded
 * shapes: the whole call is capturable.
 * dtype GBMOE_BF16: x (G, M, K) and recv_x bf16; x_scales, recv_scales
 *   ignored.
 * dtype GBMOE_FP8_E4M3 (the tokens quantised before the dispatch, as the
 *   prepare step does): x (G, M, K) e4m3 codes with x_scales (G*M, K/128)
 *   fp32, one per token and 128-group (moe_quant_fp8_group's layout), and
 *   recv_x (E, worst_tokens, K) e4m3 with recv_scales (E*worst_tokens,
 *   K/128) fp32: each row's scales travel with its codes, in the layout
 *   moe_batched_masked_experts takes for e4m3 (pass recv_scales +
 *   g*(E/G)*worst_tokens*(K/128) for shard g).  K a multiple of 128.
 * ws: moe_workspace_size(GBMOE_WS_EP_DISPATCH, M, E, G, K, topk, 0) bytes,
 * 16-byte aligned.  K a multiple of 8, E a multiple of G; x and recv_x
 * 16-byte aligned, the scales 4-byte aligned.  err_word may be NULL.  On
 * several GPUs each shard's receive block would live on its own GPU and the
 * row copies would be peer stores; this call is the single-GPU form. */
gbmoe_status_t moe_ep_dispatch(const void *x, const float *x_scales,
                               const int32_t *num_tokens, const int32_t *topk_ids,
                               int G, int M, int K, int E, int topk, int worst_tokens,
                               int dtype, void *recv_x, float *recv_scales,
                               int32_t *recv_counts, int32_t *recv_pos, void *ws,
                               size_t ws_bytes, int32_t *err_word, gbmoe_stream_t stream);

/* Expert-parallel combine of the same mode: for every shard r and valid token
 * t < num_tokens[r] (device),
 *   out[r, t, :] = bf16( sum_{j = 0 .. topk-1} topk_weights[r, t, j] *
 *                        recv_y[e_j, recv_pos[r, t, j], :] )
 * with e_j = topk_ids[r, t, j], in fp32, in slot order, skipping pairs with
 * recv_pos < 0 (TopKWeightAndReduce.apply of the modular kernel: weights
 * applied, then the reduce).  recv_y (E, worst_tokens, K) bf16 holds the
 * experts' unweighted outputs at the rows dispatch gave them (the y_b of
 * moe_batched_masked_experts).  Rows of out of padded tokens are not
 * written; the token loop is bounded by num_tokens on the device, never by M.
 * out (G, M, K) bf16, 16-byte aligned. */
gbmoe_status_t moe_ep_combine(const uint16_t *recv_y, const int32_t *topk_ids,
                              const int32_t *recv_pos, const float *topk_weights,
                              const int32_t *num_tokens, int G, int M, int K, int E,
                              int topk, int worst_tokens, uint16_t *out,
                              gbmoe_stream_t stream);

/* moe_align_permute without a workspace argument.  The pages have no
 * counterpart of this call: it exists for callers that cannot give the
 * library scratch memory -- for instance a plugin interface that hands an
 * operator only its input and output buffers, or a serving engine that has
 * carved up all device memory in advance and has no spare buffer to lend
 * per call.  It computes exactly what moe_align_permute computes with
 * expert_map = NULL and E_global = E (the routed ids are this GPU's expert
 * ids; there is no expert-map argument, so an id outside [0, E) is skipped
 * and flagged GBMOE_ERR_BAD_EXPERT_ID, never treated as off-shard), minus
 * ws / ws_bytes, and allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.
 * Its scratch (one int32 histogram of E entries per chunk of 2048 pairs) is a
 * fixed 256 KiB array in device memory that belongs to the library: every
 * GPU that loads the library keeps it until the process exits.  Limit:
 * ceil(M*topk / 2048) * E <= 65536 (for example M*topk <= 524288 pairs with
 * E = 256); larger problems return GBMOE_INVALID_ARG and enqueue nothing.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 * All calls share the one array and it keeps the last call's contents; every
 * entry a call reads is first written by the same call, so nothing needs
 * clearing.  Two calls that overlap on the GPU (different streams without
 * ordering between them) race on the array and give wrong results.
 * `stream` must belong to the current device: the array's address is looked
 * up for the current device, and a stream of another device is refused with
 * GBMOE_INVALID_ARG before anything is enqueued. */
gbmoe_status_t moe_align_permute_no_ws(const int32_t *topk_ids, int M,
                                       int topk, int E, int32_t *counts,
                                       int32_t *offsets,
                                       int32_t *sorted_pair_ids, int32_t *inv,
                                       int32_t *err_word,
                                       gbmoe_stream_t stream);

/* Self-test of the failure path of the pipeline waits.  Every wait of the
 * GEMM kernels on a pipeline barrier is bounded: after its limit it gives
 * up, ORs GBMOE_ERR_TIMEOUT into err_word and the kernel leaves its loops
 * instead of hanging.  This call runs that same bounded wait, with a limit of
 * limit_us microseconds (1 .. 1000000), on a shared-memory barrier that
 * nothing ever completes: once the stream reaches it, *err_word has the
 * GBMOE_ERR_TIMEOUT bit set after about limit_us, and the context stays
 * usable.  One launch of one 32-thread block; err_word is caller-owned
 * device memory (not cleared here).  GBMOE_INVALID_ARG for a NULL err_word
 * or a limit outside the range, before any launch. */
gbmoe_status_t gbmoe_selftest_bounded_wait(int32_t *err_word, int limit_us,
                                           gbmoe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBMOE_H */

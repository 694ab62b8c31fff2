// kernels.h -- host-side launchers of the library's kernels (internal).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gbmoe.h"

namespace gbmoe {

// route.cu
cudaError_t launch_route(const float *logits, const float *bias, int M, int E,
                         int topk, int score_fn, int n_groups, int topk_groups,
                         int renorm, int32_t *ids, float *weights,
                         cudaStream_t s);

// permute.cu
// Eg: routed (global) experts; map (Eg) global -> local id or -1 (NULL:
// identity, Eg == E); E: local experts
cudaError_t launch_count(const int32_t *ids, int P, int Eg, const int32_t *map,
                         int E, int32_t *counts, int32_t *err, int num_sms,
                         cudaStream_t s);
int align_num_chunks(int P);
cudaError_t launch_align(const int32_t *ids, int P, int Eg, const int32_t *map,
                         int E, int32_t *counts, int32_t *offsets, int32_t *sorted,
                         int32_t *inv, int32_t *chunk_hist, int32_t *err,
                         cudaStream_t s);
// out_s is group-major: (n_scales, out_s_ld); row_w (per pair, bf16 rows
// only) or NULL
cudaError_t launch_gather_rows(const void *x, const float *xs, const float *row_w,
                               int row_bytes, int n_scales, const int32_t *sorted,
                               const int32_t *total, int P, int topk,
                               void *out, float *out_s, int64_t out_s_ld,
                               int num_sms, cudaStream_t s);
// row-major (rows, G) fp32 -> group-major (G, ld), ld >= rows; G <= 128
// counts (E) and T, when counts is given: the rows are (E, T) and a run of
// 32 rows that holds no row r with r % T < clamp(counts[r / T], 0, T) is
// not moved (its scales stay as the output held them)
cudaError_t launch_scales_group_major(const float *in, int64_t rows, int G, float *out,
                                      int64_t ld, int num_sms, cudaStream_t s,
                                      const int32_t *counts = nullptr, int T = 0);
cudaError_t launch_reduce(const uint16_t *y_slot, const int32_t *inv, int M,
                          int topk, int K, uint16_t *out, int num_sms,
                          cudaStream_t s);

// ep.cu -- worst-tokens dispatch / combine over G shards in this GPU's memory
struct EpWorkspace {
  int32_t *ids_eff;     // (G*M*topk): the pairs' expert ids, E for padded tokens
  int32_t *map;         // (E + 1): e -> e, E -> -1 (skipped)
  int32_t *counts;      // (E)
  int32_t *offsets;     // (E + 1)
  int32_t *sorted;      // (G*M*topk)
  int32_t *inv;         // (G*M*topk)
  int32_t *chunk_hist;  // (align_num_chunks(G*M*topk) * E)
};
// rows of row_bytes (a multiple of 16); xs / recv_s: e4m3 group scales
// (K/128 per row) carried with the rows, or NULL
cudaError_t launch_ep_dispatch(const void *x, const float *xs, const int32_t *num_tokens,
                               const int32_t *topk_ids, int G, int M, int K, int row_bytes,
                               int E, int topk, int worst, void *recv_x, float *recv_s,
                               int32_t *recv_counts, int32_t *recv_pos, const EpWorkspace &w,
                               int32_t *err, int num_sms, cudaStream_t s);
cudaError_t launch_ep_combine(const uint16_t *recv_y, const int32_t *topk_ids,
                              const int32_t *recv_pos, const float *topk_weights,
                              const int32_t *num_tokens, int G, int M, int K, int E, int topk,
                              int worst, uint16_t *out, int num_sms, cudaStream_t s);

// quant.cu
// row_w (M) or NULL: rows multiplied by their weight (fp32) before quantising
cudaError_t launch_quant_group(const uint16_t *x, const float *row_w, int M, int K,
                               uint8_t *q, float *scales, int num_sms, cudaStream_t s);
// launch_quant_group writing its codes and scales straight to the permuted
// rows: A row inv[t*topk + j] (skipped when negative), As group-major (K/128, ld)
cudaError_t launch_quant_group_scatter(const uint16_t *x, const float *row_w, int M, int K,
                                       const int32_t *inv, int topk, uint8_t *A, float *As,
                                       int64_t ld, int num_sms, cudaStream_t s);
cudaError_t launch_quant_row(const uint16_t *x, const float *row_w, int M, int K,
                             uint8_t *q, float *scales, int num_sms, cudaStream_t s);
// launch_quant_row writing codes and the row's scale straight to the permuted
// rows: A row inv[t*topk + j] (skipped when negative), As[that row]; topk <= 32
cudaError_t launch_quant_row_scatter(const uint16_t *x, const float *row_w, int M, int K,
                                     const int32_t *inv, int topk, uint8_t *A, float *As,
                                     int num_sms, cudaStream_t s);
// static_scale (device fp32) or NULL: the codes use that scale instead of the
// tensor's maximum (amax then unused)
cudaError_t launch_quant_tensor(const uint16_t *x, const float *row_w, int M, int K,
                                const int32_t *n_rows, uint8_t *q, float *row_scales,
                                uint32_t *amax, const float *static_scale, int num_sms,
                                cudaStream_t s);
// launch_quant_tensor over all M rows of x with row t's codes and scale
// written to the permuted rows A / As [inv[t*topk + j]] (skipped when negative)
cudaError_t launch_quant_tensor_scatter(const uint16_t *x, const float *row_w, int M, int K,
                                        const int32_t *inv, int topk, uint8_t *A, float *As,
                                        uint32_t *amax, const float *static_scale, int num_sms,
                                        cudaStream_t s);
cudaError_t launch_quant_block(const uint16_t *w, int64_t R, int C, uint8_t *q,
                               float *scales, cudaStream_t s);

// gemm.cu -- grouped GEMMs on tcgen05 / TMEM fed by TMA
enum GemmMode { kGateUp = 0, kDown = 1 };

struct GroupedGemmArgs {
  int mode;                  // kGateUp or kDown
  int fp8;                   // 0: bf16 operands, 1: e4m3 with fp32 block scales
  int fp8ch;                 // 1: e4m3 with one fp32 scale per row of A and per row of B
                             //    (A_scales (a_rows), B_scales (E * rows of B per expert))
  int act;                   // gate/up: GBMOE_ACT_SILU or GBMOE_ACT_GELU
  // row groups: Standard (offsets != nullptr): expert e owns rows
  // [offsets[e], offsets[e+1]) of A.  Batched: rows [e*T, e*T + min(counts[e], T)).
  const int32_t *offsets;
  const int32_t *counts;
  int E, T;
  int N, K;                  // problem sizes (w1 (E, 2N, K), w2 (E, K, N))
  // operands
  const void *A;             // (rows, Kd) bf16 or e4m3, Kd = K (gate-up) or N (down)
  int64_t a_rows;            // rows of A's allocation
  const float *A_scales;     // fp8: (Kd/128, scale_ld), group-major
  int64_t scale_ld;          // fp8: leading dimension of A_scales / out_scales (a_rows rounded up to 4)
  const void *B;             // w1 or w2
  const float *B_scales;     // fp8: w1 (E, 2N/128, K/128) / w2 (E, K/128, N/128)
  // outputs
  void *out;                 // gate-up: H (a_rows, N); down: y rows of K bf16
  float *out_scales;         // fp8 gate-up: H scales (N/128, scale_ld), group-major
  const int32_t *sorted_pair_ids;  // down, Standard: output row = pair id
  const float *topk_weights;       // down, Standard: row scale
  int32_t *err;
};

cudaError_t launch_grouped_gemm(const GroupedGemmArgs &a, int num_sms,
                                cudaStream_t s);
// whether launch_grouped_gemm runs a bf16 launch on CTA pairs (gemm2sm.cu)
bool bf16_uses_cta_pairs(const GroupedGemmArgs &a);
// gemm2sm.cu: bf16 on CTA pairs (cta_group::2, 256 x 256 tiles)
cudaError_t launch_grouped_gemm_pair(const GroupedGemmArgs &a, int num_sms,
                                     cudaStream_t s);
// gemm_fp8.cu
cudaError_t launch_grouped_gemm_fp8(const GroupedGemmArgs &a, int num_sms,
                                    cudaStream_t s);

// api.cu: map a cudaError_t to a status, remembering it for
// gbmoe_last_cuda_error
gbmoe_status_t status_from_cuda(cudaError_t e);

// 2-D TMA tensor map (cuTensorMapEncodeTiled, resolved once through the
// runtime): `cols` x `rows` elements, rows `row_stride_bytes` apart, boxes of
// box_cols x box_rows, 128-byte swizzle or none.
enum { kTmapU8 = 0, kTmapBF16 = 1, kTmapF32 = 2 };
bool encode_tmap_2d(CUtensorMap *map, const void *base, int kind, uint64_t cols,
                    uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols,
                    uint32_t box_rows, bool swizzle128);

}  // namespace gbmoe

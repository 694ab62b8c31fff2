// ep.cu -- expert-parallel dispatch and combine in the worst-tokens mode of
// "EP: CUDA-graph-safe HT internode dispatch+combine (worst-tokens mode)"
// (uccl pull request 7, and the vLLM commit message quoted under it), for G
// shards ("ranks") whose buffers live in this GPU's memory.
//
// Every shard r holds up to M tokens (num_tokens[r] of them valid, a device
// value) with their top-k routed experts; shard g owns the experts
// [g * E / G, (g + 1) * E / G).  Dispatch sends each valid (token, slot) pair
// to the receive block of its expert, which has a static worst-case shape
// (worst_tokens rows per expert): rows are taken in ascending pair order
// (source shard, token, slot), the per-expert counts land in a device int32
// tensor (the one the masked grouped GEMM reads inside a CUDA graph), and
// the row each pair landed in is kept for the combine.  Combine sums, for
// every valid token of every shard, its slots' expert outputs weighted by the
// router weights, in slot order, in fp32, rounded once to bf16.  No host
// reads a count, no loop runs over the padded shapes (the pair loops are
// bounded by the device total of dispatched pairs and the token loops by
// num_tokens), and nothing waits on another launch or on the host, so both
// calls can be captured in a CUDA graph and replayed with fresh data.
//
// With e4m3 tokens (quantised before the dispatch, as the prepare step does)
// each row's 1 x 128 group scales travel with its codes into a receive block
// of scales laid out like the rows.
//
// The counting sort is the one of moe_align_permute (permute.cu), run over
// the concatenated pairs of all shards with padded tokens mapped to "not
// routed here" (skipped without an error).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbmoe {

namespace {

// ids_eff[p] = topk_ids[p] for pairs of valid tokens, E (an id that the map
// below sends to "skipped") for the padded ones; map[e] = e, map[E] = -1.
// The sort then sees E + 1 routed ids mapped onto E experts.
__global__ void __launch_bounds__(256)
    ep_mask_kernel(const int32_t *__restrict__ ids, const int32_t *__restrict__ num_tokens,
                   int R, int M, int topk, int E, int32_t *__restrict__ ids_eff,
                   int32_t *__restrict__ map) {
  const size_t P = (size_t)R * M * topk;
  for (size_t p = blockIdx.x * (size_t)blockDim.x + threadIdx.x; p < P;
       p += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(p / ((size_t)M * topk));
    const int t = (int)((p / topk) % M);
    const int n = min(max(__ldg(num_tokens + r), 0), M);
    const int g = __ldg(ids + p);
    // a routed id outside [0, E) becomes -1, which the sort skips and flags
    ids_eff[p] = t < n ? (g >= 0 && g < E ? g : -1) : E;
  }
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e <= E; e += gridDim.x * blockDim.x)
    map[e] = e < E ? e : -1;
}

// recv_pos[p] = row of pair p within its expert's block (-1: not
// dispatched); recv_counts[e] = min(count, worst); a count beyond the static
// worst-case shape is clamped and flagged (its extra pairs are dropped).
__global__ void __launch_bounds__(256)
    ep_positions_kernel(const int32_t *__restrict__ ids_eff, const int32_t *__restrict__ inv,
                        const int32_t *__restrict__ offsets, const int32_t *__restrict__ counts,
                        size_t P, int E, int worst, int32_t *__restrict__ recv_pos,
                        int32_t *__restrict__ recv_counts, int32_t *err) {
  for (size_t p = blockIdx.x * (size_t)blockDim.x + threadIdx.x; p < P;
       p += (size_t)gridDim.x * blockDim.x) {
    const int i = inv[p];
    int pos = -1;
    if (i >= 0) {
      const int e = ids_eff[p];
      pos = i - offsets[e];
      if (pos >= worst) pos = -1;
    }
    recv_pos[p] = pos;
  }
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    int c = counts[e];
    if (c > worst) {
      set_err(err, GBMOE_ERR_COUNT_RANGE);
      c = worst;
    }
    recv_counts[e] = c;
  }
}

// recv_x[e, pos] = x[token of pair] for the sorted positions below the
// device total offsets[E]: one warp per row, 16-byte vectors; e4m3 rows
// bring their n_scales group scales along (xs NULL: none).
__global__ void __launch_bounds__(256)
    ep_dispatch_rows_kernel(const uint4 *__restrict__ x, const float *__restrict__ xs,
                            const int32_t *__restrict__ sorted,
                            const int32_t *__restrict__ ids_eff,
                            const int32_t *__restrict__ offsets, int E, int topk, int worst,
                            int row_vecs, int n_scales, uint4 *__restrict__ recv_x,
                            float *__restrict__ recv_s) {
  const int lane = threadIdx.x & 31;
  const int total = offsets[E];
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < total;
       i += (gridDim.x * blockDim.x) >> 5) {
    const int p = sorted[i];
    const int e = ids_eff[p];
    const int pos = i - offsets[e];
    if (pos >= worst) continue;  // beyond the static shape: dropped (flagged)
    const size_t tok = (size_t)(p / topk), slot = (size_t)e * worst + pos;
    const uint4 *src = x + tok * row_vecs;
    uint4 *dst = recv_x + slot * row_vecs;
    for (int v = lane; v < row_vecs; v += 32) dst[v] = src[v];
    if (xs)
      for (int j = lane; j < n_scales; j += 32) recv_s[slot * n_scales + j] = xs[tok * n_scales + j];
  }
}

// out[r, t, :] = bf16( sum_j w[r,t,j] * recv_y[e_j, pos_j, :] ) over the
// slots j in order, fp32; tokens t >= num_tokens[r] are not touched.  One
// thread per 8 columns of a token.
__global__ void __launch_bounds__(256)
    ep_combine_kernel(const uint4 *__restrict__ recv_y, const int32_t *__restrict__ ids,
                      const int32_t *__restrict__ recv_pos, const float *__restrict__ w,
                      const int32_t *__restrict__ num_tokens, int R, int M, int topk, int E,
                      int worst, int kvec, uint4 *__restrict__ out) {
  const size_t n = (size_t)R * M * kvec;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t tok = idx / kvec;  // r * M + t
    const int c = (int)(idx % kvec);
    const int r = (int)(tok / M), t = (int)(tok % M);
    if (t >= min(max(__ldg(num_tokens + r), 0), M)) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < topk; ++j) {
      const size_t p = tok * topk + j;
      const int pos = __ldg(recv_pos + p);
      const int e = __ldg(ids + p);
      if (pos < 0 || e < 0 || e >= E) continue;
      const float wj = __ldg(w + p);
      const uint4 v = __ldg(recv_y + ((size_t)e * worst + pos) * kvec + c);
      const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        acc[2 * i] = fmaf(wj, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(wj, f.y, acc[2 * i + 1]);
      }
    }
    out[tok * kvec + c] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

int grid_for(size_t work, int per_block, int num_sms) {
  size_t b = (work + per_block - 1) / per_block;
  if (b > (size_t)8 * num_sms) b = (size_t)8 * num_sms;
  return b < 1 ? 1 : (int)b;
}

}  // namespace

cudaError_t launch_ep_dispatch(const void *x, const float *xs, const int32_t *num_tokens,
                               const int32_t *topk_ids, int R, int M, int K, int row_bytes,
                               int E, int topk, int worst, void *recv_x, float *recv_s,
                               int32_t *recv_counts, int32_t *recv_pos, const EpWorkspace &w,
                               int32_t *err, int num_sms, cudaStream_t s) {
  const size_t P = (size_t)R * M * topk;
  ep_mask_kernel<<<grid_for(P, 256, num_sms), 256, 0, s>>>(topk_ids, num_tokens, R, M, topk, E,
                                                          w.ids_eff, w.map);
  cudaError_t st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  st = launch_align(w.ids_eff, (int)P, E + 1, w.map, E, w.counts, w.offsets, w.sorted, w.inv,
                    w.chunk_hist, err, s);
  if (st != cudaSuccess) return st;
  ep_positions_kernel<<<grid_for(P, 256, num_sms), 256, 0, s>>>(
      w.ids_eff, w.inv, w.offsets, w.counts, P, E, worst, recv_pos, recv_counts, err);
  st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  ep_dispatch_rows_kernel<<<grid_for(P, 8, num_sms), 256, 0, s>>>(
      static_cast<const uint4 *>(x), xs, w.sorted, w.ids_eff, w.offsets, E, topk, worst,
      row_bytes / 16, K / 128, static_cast<uint4 *>(recv_x), recv_s);
  return cudaGetLastError();
}

cudaError_t launch_ep_combine(const uint16_t *recv_y, const int32_t *topk_ids,
                              const int32_t *recv_pos, const float *topk_weights,
                              const int32_t *num_tokens, int R, int M, int K, int E, int topk,
                              int worst, uint16_t *out, int num_sms, cudaStream_t s) {
  const size_t n = (size_t)R * M * (K / 8);
  ep_combine_kernel<<<grid_for(n, 256, num_sms), 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(recv_y), topk_ids, recv_pos, topk_weights, num_tokens, R,
      M, topk, E, worst, K / 8, reinterpret_cast<uint4 *>(out));
  return cudaGetLastError();
}

}  // namespace gbmoe

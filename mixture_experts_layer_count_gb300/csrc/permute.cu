// permute.cu -- per-expert counts, the stable counting sort of (token, slot)
// pairs by expert (offsets, sorted pair ids, inverse map), the row gather
// that feeds the first grouped GEMM, and the ordered top-k reduce.
//
// Counts: ExpertTokensMetadata.expert_num_tokens / count_expert_num_tokens in
// "vllm/model_executor/layers/fused_moe/modular_kernel.py".  Sort and gather:
// the "Permute" of [Permute-Experts-Unpermute].  Reduce: [Finalize],
// TopKWeightAndReduce.apply / FusedMoEPrepareAndFinalize.finalize.
//
// Integer work only (no floating-point atomics): every result here is
// independent of scheduling, so repeated runs are bitwise identical.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbmoe {

namespace {

constexpr int kAlignChunk = 2048;   // pairs per block in the sort
constexpr int kAlignThreads = 256;  // 8 warps
constexpr int kAlignWarps = kAlignThreads / 32;

// The local expert of a routed (global) id through expert_map (NULL: the
// identity): the local id, -1 for an expert that is not on this shard (the
// pair is skipped silently), -2 for an invalid id (skipped and flagged).
__device__ __forceinline__ int local_expert(int g, int Eg, const int32_t *__restrict__ map,
                                            int El) {
  if (g < 0 || g >= Eg) return -2;
  const int l = map ? map[g] : g;
  if (l == -1) return -1;
  return (l >= 0 && l < El) ? l : -2;
}

// ---------------------------------------------------------------- counts --

__global__ void __launch_bounds__(1024)
    count_kernel(const int32_t *__restrict__ ids, int P, int Eg,
                 const int32_t *__restrict__ map, int E,
                 int32_t *__restrict__ counts, int32_t *err) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P;
       p += gridDim.x * blockDim.x) {
    const int e = local_expert(ids[p], Eg, map, E);
    if (e >= 0)
      atomicAdd(&hist[e], 1);
    else if (e == -2)
      bad = true;
  }
  if (bad) set_err(err, GBMOE_ERR_BAD_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&counts[e], hist[e]);
}

// ---------------------------------------------------- stable counting sort --

// pass 1: histogram of each chunk of kAlignChunk pairs -> chunk_hist[b][e]
__global__ void __launch_bounds__(kAlignThreads)
    align_hist_kernel(const int32_t *__restrict__ ids, int P, int Eg,
                      const int32_t *__restrict__ map, int E,
                      int32_t *__restrict__ chunk_hist, int32_t *err) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kAlignChunk;
  const int p1 = min(P, p0 + kAlignChunk);
  bool bad = false;
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = local_expert(ids[p], Eg, map, E);
    if (e >= 0)
      atomicAdd(&hist[e], 1);
    else if (e == -2)
      bad = true;
  }
  if (bad) set_err(err, GBMOE_ERR_BAD_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// pass 2 (one block of 1024 threads, E <= 1024): counts[e] = sum over chunks;
// offsets = exclusive prefix sum of the counts; chunk_hist[b][e] becomes the
// first sorted position of chunk b's pairs of expert e.
__global__ void __launch_bounds__(1024)
    align_scan_kernel(int E, int n_chunks, int32_t *__restrict__ chunk_hist,
                      int32_t *__restrict__ counts,
                      int32_t *__restrict__ offsets) {
  __shared__ int32_t warp_tot[32];
  const int e = threadIdx.x;
  const int lane = e & 31, warp = e >> 5;
  int c = 0;
  if (e < E)
    for (int b = 0; b < n_chunks; ++b) c += chunk_hist[(size_t)b * E + e];
  // block-wide inclusive scan of c
  int x = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int incl = x + (warp > 0 ? warp_tot[warp - 1] : 0);
  const int excl = incl - c;
  if (e < E) {
    if (counts) counts[e] = c;
    offsets[e] = excl;
    int run = excl;
    for (int b = 0; b < n_chunks; ++b) {
      int h = chunk_hist[(size_t)b * E + e];
      chunk_hist[(size_t)b * E + e] = run;
      run += h;
    }
  }
  if (e == E - 1) offsets[E] = incl;
}

// pass 3: each block walks its chunk in order, 256 pairs per step; a pair's
// position = chunk base of its expert + pairs of that expert in earlier steps
// + in earlier warps of this step + in lower lanes of its warp.
__global__ void __launch_bounds__(kAlignThreads)
    align_scatter_kernel(const int32_t *__restrict__ ids, int P, int Eg,
                         const int32_t *__restrict__ map, int E,
                         const int32_t *__restrict__ chunk_base,
                         int32_t *__restrict__ sorted,
                         int32_t *__restrict__ inv) {
  extern __shared__ int32_t sm[];
  int32_t *run = sm;            // [E]
  int32_t *wcnt = sm + E;       // [kAlignWarps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) {
    run[e] = chunk_base[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < kAlignWarps; ++w) wcnt[w * E + e] = 0;
  }
  __syncthreads();
  const int p0 = blockIdx.x * kAlignChunk;
  const int p1 = min(P, p0 + kAlignChunk);
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int r0 = p0; r0 < p1; r0 += kAlignThreads) {
    const int p = r0 + tid;
    const bool in = p < p1;
    const int e = in ? local_expert(ids[p], Eg, map, E) : -1;
    const bool ok = e >= 0;
    const int key = ok ? e : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & lt_mask);
    if (ok && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (ok) {
      int pos = run[e] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w * E + e];
      sorted[pos] = p;
      inv[p] = pos;
    } else if (in) {
      inv[p] = -1;
    }
    __syncthreads();
    for (int x = tid; x < E; x += blockDim.x) {
      int s = 0;
      for (int w = 0; w < kAlignWarps; ++w) {
        s += wcnt[w * E + x];
        wcnt[w * E + x] = 0;
      }
      run[x] += s;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ gather --

// out[i] = x[sorted[i] / topk] for i < *total (one warp per row, 16-byte
// vectors); FP8 also carries the row's group scales, written group-major
// (out_s[g * out_s_ld + i]) so that a GEMM tile's scales of one K block are
// contiguous.  The scales are copied after the rows by every thread of the
// grid, one (row, 8 groups) unit at a time with the rows fastest, so that a
// warp's stores of one group cover 32 consecutive rows.  row_w (bf16 rows
// only, per pair or NULL): the row is scaled by the pair's router weight in
// fp32 and rounded back to bf16 (apply_router_weight_on_input).
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint4 *__restrict__ x, const float *__restrict__ xs,
                       const float *__restrict__ row_w, int row_vecs, int n_scales,
                       const int32_t *__restrict__ sorted,
                       const int32_t *__restrict__ total, int P, int topk,
                       uint4 *__restrict__ out, float *__restrict__ out_s,
                       int64_t out_s_ld) {
  const int lane = threadIdx.x & 31;
  const int n = min(*total, P);
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n;
       i += (gridDim.x * blockDim.x) >> 5) {
    const int pair = sorted[i];
    const int t = pair / topk;
    const uint4 *src = x + (size_t)t * row_vecs;
    uint4 *dst = out + (size_t)i * row_vecs;
    if (row_w) {
      const float w = row_w[pair];
      for (int v = lane; v < row_vecs; v += 32) {
        uint4 u = src[v];
        uint32_t *h = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(h[j] << 16) * w;
          const float hi = __uint_as_float(h[j] & 0xffff0000u) * w;
          h[j] = pack_bf16x2(lo, hi);
        }
        dst[v] = u;
      }
    } else {
      for (int v = lane; v < row_vecs; v += 32) dst[v] = src[v];
    }
  }
  if (xs) {
    const int n_units = n * ((n_scales + 7) >> 3);
    for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += gridDim.x * blockDim.x) {
      const int g0 = (u / n) << 3, i = u % n;
      const float *src = xs + (size_t)(sorted[i] / topk) * n_scales;
      float *dst = out_s + (size_t)g0 * out_s_ld + i;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        if (g0 + g < n_scales) dst[(size_t)g * out_s_ld] = src[g0 + g];
    }
  }
}

// ------------------------------------------------------------------ reduce --

// out[t, :] = bf16(sum_j y_slot[t, j, :]) in slot order, fp32 sums; one thread
// per 8 output columns.  The slots of a token are loaded B at a time (B =
// 2, 4 or 8, the smallest that covers topk, up to 8), all loads issued
// before the first add (a slot of a pair not computed on this shard -- inv
// < 0 -- is not loaded and adds +0.0, which leaves the sum bit for bit as
// skipping it would: the sum starts at +0.0 and never becomes -0.0), then
// added in slot order.
template <int B>
__global__ void __launch_bounds__(256)
    reduce_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ inv,
                  int M, int topk, int kvec, uint4 *__restrict__ out) {
  const size_t n = (size_t)M * kvec;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(idx / kvec);
    const int c = (int)(idx % kvec);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < topk; j0 += B) {
      uint4 v[B];
#pragma unroll
      for (int u = 0; u < B; ++u) {
        const int j = j0 + u;
        const int p = t * topk + j;
        const bool take = j < topk && (!inv || __ldg(inv + p) >= 0);
        v[u] = take ? __ldg(y + (size_t)p * kvec + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < B; ++u) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[u]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h[i]);
          acc[2 * i] += f.x;
          acc[2 * i + 1] += f.y;
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    out[(size_t)t * kvec + c] = o;
  }
}

// Row-major scales (rows, G) -> group-major (G, ld): 32 rows at a time
// through shared memory, so both the reads (a run of 32 * G floats) and the
// writes (32 consecutive floats of each of the G groups) are coalesced.
__global__ void __launch_bounds__(256)
    scales_group_major_kernel(const float *__restrict__ in, int64_t rows, int G,
                              float *__restrict__ out, int64_t ld,
                              const int32_t *__restrict__ counts, int T) {
  extern __shared__ float tile[];  // [32][G + 1]
  const int gp = G + 1;
  for (int64_t r0 = (int64_t)blockIdx.x * 32; r0 < rows; r0 += (int64_t)gridDim.x * 32) {
    const int nr = (int)(rows - r0 < 32 ? rows - r0 : 32);
    if (counts) {  // uniform over the block: r0 and counts are
      // rows (E, T): row r holds a token of expert r / T when r % T is below
      // that expert's count; a run of 32 rows with no such row is skipped
      bool live = false;
      if ((int)threadIdx.x < nr) {
        const int64_t r = r0 + threadIdx.x;
        const int c = __ldg(counts + r / T);
        live = r % T < (int64_t)(c < 0 ? 0 : (c > T ? T : c));
      }
      if (!__syncthreads_or(live)) continue;
    }
    for (int i = threadIdx.x; i < nr * G; i += blockDim.x)
      tile[(i / G) * gp + i % G] = in[r0 * G + i];
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * G; i += blockDim.x) {
      const int g = i >> 5, r = i & 31;
      if (r < nr) out[(int64_t)g * ld + r0 + r] = tile[r * gp + g];
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_count(const int32_t *ids, int P, int Eg, const int32_t *map,
                         int E, int32_t *counts, int32_t *err, int num_sms,
                         cudaStream_t s) {
  cudaError_t st = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
  if (st != cudaSuccess) return st;
  int blocks = (P + 1023) / 1024;
  if (blocks > 2 * num_sms) blocks = 2 * num_sms;
  if (blocks < 1) blocks = 1;
  count_kernel<<<blocks, 1024, sizeof(int32_t) * E, s>>>(ids, P, Eg, map, E, counts, err);
  return cudaGetLastError();
}

int align_num_chunks(int P) { return (P + kAlignChunk - 1) / kAlignChunk; }

cudaError_t launch_align(const int32_t *ids, int P, int Eg, const int32_t *map,
                         int E, int32_t *counts, int32_t *offsets, int32_t *sorted,
                         int32_t *inv, int32_t *chunk_hist, int32_t *err,
                         cudaStream_t s) {
  const int nb = align_num_chunks(P);
  if (nb > 0) {
    align_hist_kernel<<<nb, kAlignThreads, sizeof(int32_t) * E, s>>>(ids, P, Eg, map, E,
                                                                    chunk_hist, err);
  }
  align_scan_kernel<<<1, 1024, 0, s>>>(E, nb, chunk_hist, counts, offsets);
  if (nb > 0) {
    const size_t smem = sizeof(int32_t) * (size_t)E * (1 + kAlignWarps);
    align_scatter_kernel<<<nb, kAlignThreads, smem, s>>>(ids, P, Eg, map, E, chunk_hist,
                                                         sorted, inv);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void *x, const float *xs, const float *row_w,
                               int row_bytes, int n_scales, const int32_t *sorted,
                               const int32_t *total, int P, int topk,
                               void *out, float *out_s, int64_t out_s_ld,
                               int num_sms, cudaStream_t s) {
  const int warps_per_block = 8;
  int blocks = (P + warps_per_block - 1) / warps_per_block;
  if (blocks > 8 * num_sms) blocks = 8 * num_sms;
  if (blocks < 1) blocks = 1;
  gather_rows_kernel<<<blocks, 32 * warps_per_block, 0, s>>>(
      static_cast<const uint4 *>(x), xs, row_w, row_bytes / 16, n_scales, sorted,
      total, P, topk, static_cast<uint4 *>(out), out_s, out_s_ld);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const uint16_t *y_slot, const int32_t *inv, int M,
                          int topk, int K, uint16_t *out, int num_sms,
                          cudaStream_t s) {
  const int kvec = K / 8;
  const size_t n = (size_t)M * kvec;
  size_t blocks = (n + 255) / 256;
  if (blocks > (size_t)8 * num_sms) blocks = (size_t)8 * num_sms;
  if (blocks < 1) blocks = 1;
  const uint4 *y = reinterpret_cast<const uint4 *>(y_slot);
  uint4 *o = reinterpret_cast<uint4 *>(out);
  if (topk <= 2)
    reduce_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(y, inv, M, topk, kvec, o);
  else if (topk <= 4)
    reduce_kernel<4><<<(unsigned)blocks, 256, 0, s>>>(y, inv, M, topk, kvec, o);
  else
    reduce_kernel<8><<<(unsigned)blocks, 256, 0, s>>>(y, inv, M, topk, kvec, o);
  return cudaGetLastError();
}

cudaError_t launch_scales_group_major(const float *in, int64_t rows, int G, float *out,
                                      int64_t ld, int num_sms, cudaStream_t s,
                                      const int32_t *counts, int T) {
  int64_t blocks = (rows + 31) / 32;
  if (blocks > 4 * num_sms) blocks = 4 * num_sms;
  if (blocks < 1) blocks = 1;
  scales_group_major_kernel<<<(int)blocks, 256, (size_t)32 * (G + 1) * 4, s>>>(
      in, rows, G, out, ld, counts, counts ? T : 1);
  return cudaGetLastError();
}

}  // namespace gbmoe

// quant.cu -- [Quantize-Prepare] FP8 e4m3 quantisation.
//
// FusedMoEPrepareAndFinalize.prepare in
// "vllm/model_executor/layers/fused_moe/modular_kernel.py" quantises the
// activations before the experts run (per_act_token_quant / block_shape of the
// quant config).  Rule for one group (128 consecutive values of a token, or a
// 128 x 128 tile of a weight matrix):
//     s = max(amax, 1e-12) / 448       (fp32, IEEE division)
//     q = e4m3(x / s)                  (IEEE division, round to nearest even,
//                                       saturating at +-448)
// The group is 128 values, or a whole row (one scale per token of the
// activations, per_act_token_quant; per output channel of a weight matrix,
// per_out_ch_quant), or a whole tensor (per-tensor activation scale: a
// grid-wide maximum first, then the codes).
// HBM-bound: each kernel reads its input once (the row kernel a second time
// from L1/L2) and writes q and s once.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbmoe {

namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t e4m3_of(float v) {
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float group_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
}

// one half-warp per (token, 128-group): 8 values (one 16-byte load) per lane,
// two groups per warp; each warp takes two pairs of groups per loop turn
// with both loads issued first (more bytes in flight per SM)
// the codes of one lane's 8 values and the group's scale (valid when live)
__device__ __forceinline__ void quant_group_codes(const uint4 &raw, bool live, const float *row_w,
                                                  size_t t, uint2 &code, float &scale) {
  float f[8];
  float amax = 0.0f;
  const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_float(u[i] & 0xffffu);
    f[2 * i + 1] = bf16_bits_to_float(u[i] >> 16);
  }
  if (row_w) {  // apply_router_weight_on_input: the fp32 product is quantised
    const float w8 = live ? row_w[t] : 1.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], w8);
  }
  if (live) {
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1)  // within each half-warp
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  scale = 1.0f;
  code = make_uint2(0u, 0u);
  if (live) {
    const float s = group_scale(amax);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = e4m3_of(__fdiv_rn(f[i], s));
    code = make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24),
                      c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
    scale = s;
  }
}

__device__ __forceinline__ void quant_group_pair(const uint4 &raw, bool live, const float *row_w,
                                                 size_t t, size_t g, size_t vec, int hl, int G,
                                                 uint2 *__restrict__ q, float *__restrict__ scales) {
  uint2 code;
  float s;
  quant_group_codes(raw, live, row_w, t, code, s);
  if (live) {
    q[vec] = code;
    if (hl == 0) scales[t * G + g] = s;
  }
}

// the same codes sent straight to the permuted rows of the token's pairs
// (the gather of moe_permute_rows folded in): row inv[t * topk + j] of A,
// skipped when negative, gets the group's 128 codes and As[g * ld + row]
// its scale
__device__ __forceinline__ void quant_group_scatter(const uint4 &raw, bool live,
                                                    const float *row_w, size_t t, size_t g,
                                                    int hl, int K, const int32_t *__restrict__ inv,
                                                    int topk, uint2 *__restrict__ A,
                                                    float *__restrict__ As, int64_t ld) {
  uint2 code;
  float s;
  quant_group_codes(raw, live, row_w, t, code, s);
  if (!live) return;
  for (int j = 0; j < topk; ++j) {
    const int i = __ldg(inv + t * topk + j);
    if (i < 0) continue;
    A[((size_t)i * K + g * 128) / 8 + hl] = code;
    if (hl == 0) As[(size_t)g * ld + i] = s;
  }
}

__global__ void __launch_bounds__(256)
    quant_group_kernel(const uint4 *__restrict__ x, const float *__restrict__ row_w,
                       int M, int K, uint2 *__restrict__ q,
                       float *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int G = K / 128;
  const size_t n = (size_t)M * G;  // groups
  const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
  for (size_t w = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; 2 * w < n; w += 2 * nw) {
    const size_t gi0 = 2 * w + half, gi1 = 2 * (w + nw) + half;
    const bool live0 = gi0 < n, live1 = gi1 < n;
    const size_t t0 = live0 ? gi0 / G : 0, g0 = live0 ? gi0 % G : 0;
    const size_t t1 = live1 ? gi1 / G : 0, g1 = live1 ? gi1 % G : 0;
    const size_t v0 = (t0 * K + g0 * 128) / 8 + hl, v1 = (t1 * K + g1 * 128) / 8 + hl;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 r0 = live0 ? x[v0] : z;
    const uint4 r1 = live1 ? x[v1] : z;
    quant_group_pair(r0, live0, row_w, t0, g0, v0, hl, G, q, scales);
    if (2 * (w + nw) < n)  // uniform over the warp
      quant_group_pair(r1, live1, row_w, t1, g1, v1, hl, G, q, scales);
  }
}

__global__ void __launch_bounds__(256)
    quant_group_scatter_kernel(const uint4 *__restrict__ x, const float *__restrict__ row_w,
                               int M, int K, const int32_t *__restrict__ inv, int topk,
                               uint2 *__restrict__ A, float *__restrict__ As, int64_t ld) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int G = K / 128;
  const size_t n = (size_t)M * G;  // groups
  const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
  for (size_t w = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; 2 * w < n; w += 2 * nw) {
    const size_t gi0 = 2 * w + half, gi1 = 2 * (w + nw) + half;
    const bool live0 = gi0 < n, live1 = gi1 < n;
    const size_t t0 = live0 ? gi0 / G : 0, g0 = live0 ? gi0 % G : 0;
    const size_t t1 = live1 ? gi1 / G : 0, g1 = live1 ? gi1 % G : 0;
    const size_t v0 = (t0 * K + g0 * 128) / 8 + hl, v1 = (t1 * K + g1 * 128) / 8 + hl;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 r0 = live0 ? x[v0] : z;
    const uint4 r1 = live1 ? x[v1] : z;
    quant_group_scatter(r0, live0, row_w, t0, g0, hl, K, inv, topk, A, As, ld);
    if (2 * (w + nw) < n)  // uniform over the warp
      quant_group_scatter(r1, live1, row_w, t1, g1, hl, K, inv, topk, A, As, ld);
  }
}

// one warp per row, the group being the whole row: the row maximum, then
// the codes (the row is read again, from L1/L2); 8 values per 16-byte load.
// SCATTER: the codes and the scale go straight to the permuted rows of the
// token's pairs (the gather of moe_permute_rows folded in): row
// inv[t * topk + j] of q, skipped when negative, and scales[that row].
template <bool SCATTER>
__global__ void __launch_bounds__(256)
    quant_row_kernel(const uint4 *__restrict__ x, const float *__restrict__ row_w, int M,
                     int K, uint2 *__restrict__ q, float *__restrict__ scales,
                     const int32_t *__restrict__ inv, int topk) {
  const int lane = threadIdx.x & 31;
  const int vecs = K / 8;
  for (size_t t = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; t < (size_t)M;
       t += ((size_t)gridDim.x * blockDim.x) >> 5) {
    const float w = row_w ? row_w[t] : 1.0f;
    const uint4 *xr = x + t * vecs;
    float amax = 0.0f;
    for (int v = lane; v < vecs; v += 32) {
      const uint4 raw = xr[v];
      const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a = bf16_bits_to_float(u[i] & 0xffffu), b = bf16_bits_to_float(u[i] >> 16);
        if (row_w) {
          a = __fmul_rn(a, w);
          b = __fmul_rn(b, w);
        }
        amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = group_scale(amax);
    // SCATTER: lane j < topk holds the row of pair j (topk <= 32)
    const int my_dst = SCATTER && lane < topk ? __ldg(inv + t * topk + lane) : -1;
    for (int v0 = 0; v0 < vecs; v0 += 32) {  // uniform over the warp (the shuffles below)
      const int v = v0 + lane;
      const bool live = v < vecs;
      uint2 code = make_uint2(0u, 0u);
      if (live) {
        const uint4 raw = xr[v];
        const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a = bf16_bits_to_float(u[i] & 0xffffu), b = bf16_bits_to_float(u[i] >> 16);
          if (row_w) {
            a = __fmul_rn(a, w);
            b = __fmul_rn(b, w);
          }
          c[2 * i] = e4m3_of(__fdiv_rn(a, s));
          c[2 * i + 1] = e4m3_of(__fdiv_rn(b, s));
        }
        code = make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24),
                          c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
      }
      if (SCATTER) {
        for (int j = 0; j < topk; ++j) {
          const int dst = __shfl_sync(0xffffffffu, my_dst, j);
          if (live && dst >= 0) q[(size_t)dst * vecs + v] = code;
        }
      } else if (live) {
        q[t * vecs + v] = code;
      }
    }
    if (SCATTER) {
      if (my_dst >= 0) scales[my_dst] = s;
    } else if (lane == 0) {
      scales[t] = s;
    }
  }
}

// 8 values of a 16-byte vector, times the row weight (an fp32 product)
__device__ __forceinline__ void unpack8(uint4 raw, const float *row_w, size_t t, float (&v)[8]) {
  const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
  const float w = row_w ? row_w[t] : 1.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_float(u[i] & 0xffffu);
    v[2 * i + 1] = bf16_bits_to_float(u[i] >> 16);
    if (row_w) {
      v[2 * i] = __fmul_rn(v[2 * i], w);
      v[2 * i + 1] = __fmul_rn(v[2 * i + 1], w);
    }
  }
}

__device__ __forceinline__ int tensor_rows(const int32_t *n_rows, int M) {
  if (!n_rows) return M;
  const int n = *n_rows;
  return n < 0 ? 0 : (n > M ? M : n);
}

// per-tensor maximum of |v| over rows t < n: each block reduces its share,
// then one integer atomicMax on the bit pattern (a float >= 0 orders like
// its bits; max does not depend on the order of the updates)
__global__ void __launch_bounds__(256)
    quant_tensor_max_kernel(const uint4 *__restrict__ x, const float *__restrict__ row_w,
                            int M, int K, const int32_t *__restrict__ n_rows,
                            unsigned int *__restrict__ amax) {
  __shared__ float red[8];
  const int vecs = K / 8;
  const size_t total = (size_t)tensor_rows(n_rows, M) * vecs;
  float m = 0.0f;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    float v[8];
    unpack8(x[i], row_w, i / vecs, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) b = fmaxf(b, red[w]);
    atomicMax(amax, __float_as_uint(b));
  }
}

// the codes with the tensor's scale -- from its maximum, or the caller's
// static scale when given; row_scales[t] = s for every row t < n.
// SCATTER: row t's codes and scale go to the permuted rows of its pairs
// instead, q / row_scales [inv[t * topk + j]] (skipped when negative).
template <bool SCATTER>
__global__ void __launch_bounds__(256)
    quant_tensor_kernel(const uint4 *__restrict__ x, const float *__restrict__ row_w, int M,
                        int K, const int32_t *__restrict__ n_rows,
                        const unsigned int *__restrict__ amax,
                        const float *__restrict__ static_scale, uint2 *__restrict__ q,
                        float *__restrict__ row_scales, const int32_t *__restrict__ inv,
                        int topk) {
  const int vecs = K / 8;
  const size_t total = (size_t)tensor_rows(n_rows, M) * vecs;
  const float s = static_scale ? *static_scale : group_scale(__uint_as_float(*amax));
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / vecs;
    float v[8];
    unpack8(x[i], row_w, t, v);
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = e4m3_of(__fdiv_rn(v[j], s));
    const uint2 code = make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24),
                                  c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
    if (SCATTER) {
      const size_t vi = i - t * vecs;
      for (int j = 0; j < topk; ++j) {
        const int dst = __ldg(inv + t * topk + j);
        if (dst < 0) continue;
        q[(size_t)dst * vecs + vi] = code;
        if (vi == 0) row_scales[dst] = s;
      }
    } else {
      q[i] = code;
      if (i % vecs == 0) row_scales[t] = s;
    }
  }
}

// one block of 256 threads per 128 x 128 tile; thread i reads rows
// (i / 16) + 16 r, r < 8, columns (i % 16) * 8 .. + 8
__global__ void __launch_bounds__(256)
    quant_block_kernel(const uint4 *__restrict__ w, int64_t R, int C,
                       uint2 *__restrict__ q, float *__restrict__ scales) {
  __shared__ float red[8];
  const int BC = C / 128;
  const int64_t tile = blockIdx.x;
  const int64_t br = tile / BC;
  const int bc = (int)(tile % BC);
  const int tid = threadIdx.x;
  const int cvec = C / 8;  // 16-byte vectors per row
  float f[8][8];
  float amax = 0.0f;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t row = br * 128 + tid / 16 + 16 * r;
    uint4 v = w[row * cvec + bc * 16 + (tid % 16)];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[r][2 * i] = bf16_bits_to_float(u[i] & 0xffffu);
      f[r][2 * i + 1] = bf16_bits_to_float(u[i] >> 16);
      amax = fmaxf(amax, fmaxf(fabsf(f[r][2 * i]), fabsf(f[r][2 * i + 1])));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = group_scale(amax);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t row = br * 128 + tid / 16 + 16 * r;
    uint2 o;
    o.x = e4m3_of(__fdiv_rn(f[r][0], s)) | (e4m3_of(__fdiv_rn(f[r][1], s)) << 8) |
          (e4m3_of(__fdiv_rn(f[r][2], s)) << 16) | (e4m3_of(__fdiv_rn(f[r][3], s)) << 24);
    o.y = e4m3_of(__fdiv_rn(f[r][4], s)) | (e4m3_of(__fdiv_rn(f[r][5], s)) << 8) |
          (e4m3_of(__fdiv_rn(f[r][6], s)) << 16) | (e4m3_of(__fdiv_rn(f[r][7], s)) << 24);
    q[row * cvec + bc * 16 + (tid % 16)] = o;
  }
  if (tid == 0) scales[br * BC + bc] = s;
}

}  // namespace

cudaError_t launch_quant_group(const uint16_t *x, const float *row_w, int M, int K,
                               uint8_t *q, float *scales, int num_sms, cudaStream_t s) {
  const size_t warps = ((size_t)M * (K / 128) + 1) / 2;  // two groups per warp
  size_t blocks = (warps + 7) / 8;
  const size_t resident = (size_t)num_sms * 8;  // grid-stride over what is left
  if (blocks > resident) blocks = resident;
  if (blocks < 1) blocks = 1;
  quant_group_kernel<<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), row_w, M, K, reinterpret_cast<uint2 *>(q), scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_group_scatter(const uint16_t *x, const float *row_w, int M, int K,
                                       const int32_t *inv, int topk, uint8_t *A, float *As,
                                       int64_t ld, int num_sms, cudaStream_t s) {
  const size_t warps = ((size_t)M * (K / 128) + 1) / 2;
  size_t blocks = (warps + 7) / 8;
  const size_t resident = (size_t)num_sms * 8;
  if (blocks > resident) blocks = resident;
  if (blocks < 1) blocks = 1;
  quant_group_scatter_kernel<<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), row_w, M, K, inv, topk, reinterpret_cast<uint2 *>(A),
      As, ld);
  return cudaGetLastError();
}

cudaError_t launch_quant_row(const uint16_t *x, const float *row_w, int M, int K,
                             uint8_t *q, float *scales, int num_sms, cudaStream_t s) {
  size_t blocks = ((size_t)M + 7) / 8;
  const size_t resident = (size_t)num_sms * 8;
  if (blocks > resident) blocks = resident;
  if (blocks < 1) blocks = 1;
  quant_row_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), row_w, M, K, reinterpret_cast<uint2 *>(q),
      scales, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_quant_row_scatter(const uint16_t *x, const float *row_w, int M, int K,
                                     const int32_t *inv, int topk, uint8_t *A, float *As,
                                     int num_sms, cudaStream_t s) {
  if (topk < 1 || topk > 32) return cudaErrorInvalidValue;
  size_t blocks = ((size_t)M + 7) / 8;
  const size_t resident = (size_t)num_sms * 8;
  if (blocks > resident) blocks = resident;
  if (blocks < 1) blocks = 1;
  quant_row_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), row_w, M, K, reinterpret_cast<uint2 *>(A), As, inv,
      topk);
  return cudaGetLastError();
}

cudaError_t launch_quant_tensor(const uint16_t *x, const float *row_w, int M, int K,
                                const int32_t *n_rows, uint8_t *q, float *row_scales,
                                uint32_t *amax, const float *static_scale, int num_sms,
                                cudaStream_t s) {
  const size_t vecs = (size_t)M * (K / 8);
  size_t blocks = (vecs + 255) / 256;
  const size_t cap = (size_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t st;
  if (!static_scale) {  // the dynamic scale: the tensor's maximum first
    st = cudaMemsetAsync(amax, 0, sizeof(uint32_t), s);
    if (st != cudaSuccess) return st;
    quant_tensor_max_kernel<<<(unsigned)blocks, 256, 0, s>>>(
        reinterpret_cast<const uint4 *>(x), row_w, M, K, n_rows, amax);
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  quant_tensor_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), row_w, M, K, n_rows, amax, static_scale,
      reinterpret_cast<uint2 *>(q), row_scales, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_quant_tensor_scatter(const uint16_t *x, const float *row_w, int M, int K,
                                        const int32_t *inv, int topk, uint8_t *A, float *As,
                                        uint32_t *amax, const float *static_scale, int num_sms,
                                        cudaStream_t s) {
  const size_t vecs = (size_t)M * (K / 8);
  size_t blocks = (vecs + 255) / 256;
  const size_t cap = (size_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t st;
  if (!static_scale) {
    st = cudaMemsetAsync(amax, 0, sizeof(uint32_t), s);
    if (st != cudaSuccess) return st;
    quant_tensor_max_kernel<<<(unsigned)blocks, 256, 0, s>>>(
        reinterpret_cast<const uint4 *>(x), row_w, M, K, nullptr, amax);
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  quant_tensor_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), row_w, M, K, nullptr, amax, static_scale,
      reinterpret_cast<uint2 *>(A), As, inv, topk);
  return cudaGetLastError();
}

cudaError_t launch_quant_block(const uint16_t *w, int64_t R, int C, uint8_t *q,
                               float *scales, cudaStream_t s) {
  const int64_t tiles = (R / 128) * (C / 128);
  quant_block_kernel<<<(unsigned)tiles, 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(w), R, C, reinterpret_cast<uint2 *>(q),
      scales);
  return cudaGetLastError();
}

}  // namespace gbmoe

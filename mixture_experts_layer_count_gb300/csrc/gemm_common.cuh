// gemm_common.cuh -- pieces shared by the bf16 and FP8 grouped GEMM kernels:
// tile geometry, the device-side tile table (which expert, m-tile and n-tile
// a persistent CTA's i-th tile is), and small epilogue helpers.
#pragma once

#include <cuda_fp8.h>

#include "ptx.cuh"

namespace gbmoe {
namespace gemm {

constexpr int kGateUpMode = 0;
constexpr int kDownMode = 1;

constexpr int kBM = 128;     // rows per tile (UMMA M)
constexpr int kBN = 256;     // output columns per tile (UMMA N)
constexpr int kBKB = 128;    // K bytes per stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBKB;  // 16 KB
constexpr int kBStage = kBN * kBKB;  // 32 KB
constexpr int kMaxE = 512;

// Rows of expert e: Standard format [offsets[e], offsets[e+1]); Batched
// format [e*T, e*T + min(max(counts[e], 0), T)); dense (offsets and counts
// both NULL: every expert has all T rows, as the shared expert does)
// [e*T, e*T + T).  Fills rbase / rcnt and
// prefix[e+1] = tiles of expert e (m-tiles x n_tiles).  All threads of the
// block take part; a __syncthreads must follow before tile_table_scan.
__device__ __forceinline__ void tile_table_fill(const int32_t *offsets,
                                                const int32_t *counts, int E,
                                                int T, int n_tiles, int *prefix,
                                                int *rbase, int *rcnt,
                                                int32_t *err, int bm = kBM) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int b, r;
    if (offsets) {
      b = offsets[e];
      r = offsets[e + 1] - b;
    } else {
      r = counts ? counts[e] : T;
      if (r < 0 || r > T) {
        if (blockIdx.x == 0) set_err(err, GBMOE_ERR_COUNT_RANGE);
        r = r < 0 ? 0 : T;
      }
      b = e * T;
    }
    rbase[e] = b;
    rcnt[e] = r;
    prefix[e + 1] = ((r + bm - 1) / bm) * n_tiles;
  }
}

// One warp turns prefix[1..E] into inclusive prefix sums (prefix[0] = 0).
__device__ __forceinline__ void tile_table_scan(int *prefix, int E, int lane) {
  int carry = 0;
  for (int c0 = 0; c0 < E; c0 += 32) {
    const int idx = c0 + lane;
    int v = idx < E ? prefix[idx + 1] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += y;
    }
    if (idx < E) prefix[idx + 1] = v + carry;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) prefix[0] = 0;
}

// tile -> (expert, m-tile, n-tile); tiles of an expert are ordered n-major,
// m fastest, so CTAs running at the same time share weight tiles in L2.
__device__ __forceinline__ void decode_tile(const int *prefix, int E,
                                            int n_tiles, int tile, int &e,
                                            int &mt, int &nt) {
  int lo = 0, hi = E;  // prefix[lo] <= tile < prefix[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (prefix[mid] <= tile) lo = mid;
    else hi = mid;
  }
  e = lo;
  const int local = tile - prefix[e];
  const int mtiles = (prefix[e + 1] - prefix[e]) / n_tiles;
  nt = local / mtiles;
  mt = local - nt * mtiles;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// exact (erf) GELU, the "gelu" of gelu_and_mul
__device__ __forceinline__ float gelu_f(float g) {
  return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f));
}

constexpr int kActSilu = 0;
constexpr int kActGelu = 1;

template <int ACT>
__device__ __forceinline__ float gate_act(float g) {
  return ACT == kActGelu ? gelu_f(g) : silu_f(g);
}

// the same with SiLU's division by the approximate __fdividef (within 2 ulp;
// 0 for a denominator above 2^126, the limit of z / (1 + e^-z) there), for
// epilogues whose result is requantised to e4m3 next
template <int ACT>
__device__ __forceinline__ float gate_act_fast(float g) {
  return ACT == kActGelu ? gelu_f(g) : __fdividef(g, 1.0f + __expf(-g));
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3) |
         ((uint32_t)__nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3) << 8) |
         ((uint32_t)__nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3) << 16) |
         ((uint32_t)__nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3) << 24);
}

}  // namespace gemm
}  // namespace gbmoe

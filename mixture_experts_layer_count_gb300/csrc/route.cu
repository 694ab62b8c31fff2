// route.cu -- [Router]: one warp per token, top-k by warp-shuffle argmax.
//
// Softmax router: the top-k of the raw logits (softmax is increasing), weight
// softmax(l)_e, renormalised over the chosen experts on request.
// Sigmoid grouped router (DeepSeek-V3-shaped workloads): v_e = l_e + b_e;
// experts ranked by v (the order of sigmoid(v)); E experts in n_groups
// contiguous groups; a group's key is the fp32 sum of the fp32-rounded fp64
// sigmoids of its two largest v; the topk_groups best groups are kept and the
// topk best experts among them chosen; weight sigmoid(v_e), renormalised on
// request.  Equal keys go to the lower index everywhere.  The group choice
// is made on fp32 estimates of the keys and confirmed by their margin; the
// fp64 keys are computed only for a token whose cut is closer than that.
#include <cfloat>
#include <climits>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace gbmoe {

namespace {

constexpr uint32_t kFull = 0xffffffffu;

// the group-key score: fp64 sigmoid rounded once to fp32
__device__ __forceinline__ float key_sigmoid(float v) {
  return (float)(1.0 / (1.0 + exp(-(double)v)));
}

// an fp32 estimate of key_sigmoid: expf (within its documented few-ulp
// bound), one add, one IEEE division -- within ~4e-7 of key_sigmoid, so a
// key (a sum of two scores, rounded) is within ~1.1e-6 of the exact key
__device__ __forceinline__ float key_sigmoid_fp32(float v) { return 1.0f / (1.0f + expf(-v)); }

// the group selection taken from the fp32 keys stands when the last kept
// key leads the best dropped one by more than this (several times twice the
// estimate's error); otherwise the keys are recomputed exactly
constexpr float kKeyMargin = 8e-6f;

// warp-wide argmax; equal values go to the lower index
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ov = __shfl_xor_sync(kFull, v, off);
    int oi = __shfl_xor_sync(kFull, i, off);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}

// the topk_groups best groups by key (lanes < n_groups hold one key each);
// *margin = last kept key minus best dropped key
__device__ __forceinline__ uint32_t select_groups(float my_key, int lane, int n_groups,
                                                  int topk_groups, float *margin) {
  uint32_t gmask = 0;
  float last = INFINITY;
  for (int r = 0; r < topk_groups; ++r) {
    const bool cand = lane < n_groups && !((gmask >> lane) & 1u);
    float kv = cand ? my_key : -INFINITY;
    int ki = cand ? lane : INT_MAX;
    warp_argmax(kv, ki);
    if (ki < 32) gmask |= 1u << ki;
    last = kv;
  }
  const bool rest = lane < n_groups && !((gmask >> lane) & 1u);
  float kv = rest ? my_key : -INFINITY;
  int ki = rest ? lane : INT_MAX;
  warp_argmax(kv, ki);
  *margin = last - kv;
  return gmask;
}

// VPL values per lane: expert e = i * 32 + lane lives in lane (e & 31), slot
// (e >> 5), so a row of logits is read with coalesced loads.
template <int VPL>
__global__ void __launch_bounds__(256)
    route_kernel(const float *__restrict__ logits,
                 const float *__restrict__ bias, int M, int E, int topk,
                 int score_fn, int n_groups, int topk_groups, int renorm,
                 int32_t *__restrict__ ids, float *__restrict__ weights) {
  const int lane = threadIdx.x & 31;
  const int tok = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  if (tok >= M) return;  // uniform over the warp
  const float *row = logits + (size_t)tok * E;
  const bool sigmoid = score_fn == GBMOE_SIGMOID;

  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int e = i * 32 + lane;
    v[i] = -INFINITY;
    if (e < E) v[i] = row[e] + ((sigmoid && bias) ? bias[e] : 0.0f);
  }

  // ---- group limit (sigmoid only): lane g ends up holding the two largest
  // v of group g and computes the group's key itself, so the warp issues the
  // fp64 sigmoid sequence twice in all rather than twice per group (the fp64
  // pipe is narrow: a warp-wide fp64 instruction costs the same with one
  // lane active as with 32)
  const int gs = E / (n_groups > 0 ? n_groups : 1);
  int grp[VPL];  // the group of each value this lane holds (one division each)
#pragma unroll
  for (int i = 0; i < VPL; ++i) grp[i] = (i * 32 + lane) / gs;
  uint32_t gmask = kFull;
  if (sigmoid && n_groups > 1 && topk_groups < n_groups) {
    float my_t1 = -INFINITY, my_t2 = -INFINITY;
    for (int g = 0; g < n_groups; ++g) {
      float t1 = -INFINITY, t2 = -INFINITY;  // two largest v of group g
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        int e = i * 32 + lane;
        if (e < E && grp[i] == g) {
          float x = v[i];
          if (x > t1) {
            t2 = t1;
            t1 = x;
          } else if (x > t2) {
            t2 = x;
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        float o1 = __shfl_xor_sync(kFull, t1, off);
        float o2 = __shfl_xor_sync(kFull, t2, off);
        float hi = fmaxf(t1, o1);
        float lo = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
        t1 = hi;
        t2 = lo;
      }
      if (lane == g) {
        my_t1 = t1;
        my_t2 = t2;
      }
    }
    // fp32 keys first; the fp64 keys (the definition) only when two groups
    // at the cut are too close for the estimate to order them
    float my_key = -INFINITY;
    if (lane < n_groups)
      my_key = gs >= 2 ? key_sigmoid_fp32(my_t1) + key_sigmoid_fp32(my_t2)
                       : key_sigmoid_fp32(my_t1);
    float margin;
    gmask = select_groups(my_key, lane, n_groups, topk_groups, &margin);
    if (!(margin > kKeyMargin)) {  // uniform over the warp (also for NaN)
      if (lane < n_groups)
        my_key = gs >= 2 ? key_sigmoid(my_t1) + key_sigmoid(my_t2) : key_sigmoid(my_t1);
      gmask = select_groups(my_key, lane, n_groups, topk_groups, &margin);
    }
  }

  // ---- top-k experts among the eligible ones, descending
  uint32_t taken = 0;
  int my_id = -1;
  float my_v = -INFINITY;
  for (int j = 0; j < topk; ++j) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      int e = i * 32 + lane;
      if (e < E && !((taken >> i) & 1u) && ((gmask >> grp[i]) & 1u)) {
        if (bi == INT_MAX || v[i] > bv) {  // i ascending: keeps the lower e on ties
          bv = v[i];
          bi = e;
        }
      }
    }
    warp_argmax(bv, bi);
    if (bi != INT_MAX && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_id = bi;
      my_v = bv;
    }
  }

  // ---- weights
  float w = 0.0f;
  if (!sigmoid) {
    float lmax = __shfl_sync(kFull, my_v, 0);  // the first pick is the row max
    float ex = lane < topk ? __expf(my_v - lmax) : 0.0f;
    float denom;
    if (renorm) {
      denom = warp_sum(ex);
    } else {
      float part = 0.0f;
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (i * 32 + lane < E) part += __expf(v[i] - lmax);
      denom = warp_sum(part);
    }
    w = ex / denom;
  } else {
    float s = lane < topk ? 1.0f / (1.0f + __expf(-my_v)) : 0.0f;
    float denom = renorm ? warp_sum(s) : 1.0f;
    w = s / denom;
  }
  if (lane < topk) {
    ids[(size_t)tok * topk + lane] = my_id;
    weights[(size_t)tok * topk + lane] = w;
  }
}

}  // namespace

cudaError_t launch_route(const float *logits, const float *bias, int M, int E,
                         int topk, int score_fn, int n_groups, int topk_groups,
                         int renorm, int32_t *ids, float *weights,
                         cudaStream_t s) {
  const int threads = 256;
  const int blocks = (int)(((size_t)M * 32 + threads - 1) / threads);
  int vpl = (E + 31) / 32;
#define GBMOE_ROUTE(V)                                                        \
  route_kernel<V><<<blocks, threads, 0, s>>>(logits, bias, M, E, topk,       \
                                             score_fn, n_groups, topk_groups, \
                                             renorm, ids, weights)
  if (vpl <= 1) GBMOE_ROUTE(1);
  else if (vpl <= 2) GBMOE_ROUTE(2);
  else if (vpl <= 4) GBMOE_ROUTE(4);
  else if (vpl <= 8) GBMOE_ROUTE(8);
  else GBMOE_ROUTE(16);
#undef GBMOE_ROUTE
  return cudaGetLastError();
}

}  // namespace gbmoe

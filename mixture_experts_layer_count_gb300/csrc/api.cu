// api.cu -- the extern "C" entry points declared in gbmoe.h: argument
// validation, workspace carving and kernel launches.  No device memory is
// allocated here and the host is never synchronised.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gbmoe.h"
#include "kernels.h"

namespace gbmoe {
namespace {

constexpr int kMaxExperts = 512;
constexpr int kMaxTopk = 32;
constexpr size_t kWsAlign = 256;

thread_local int g_last_cuda_error = 0;

struct DeviceInfo {
  int checked = 0;  // 0: not yet, 1: supported, -1: not supported
  int num_sms = 0;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

// The kernels are compiled for sm_103a only.
gbmoe_status_t device_info(int *num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBMOE_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo &d = g_dev[dev];
  if (d.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    d.checked = (major == 10 && minor == 3 && sms > 0) ? 1 : -1;
    d.num_sms = sms;
  }
  if (d.checked < 0) return GBMOE_UNSUPPORTED;
  *num_sms = d.num_sms;
  return GBMOE_OK;
}

gbmoe_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return GBMOE_OK;
  g_last_cuda_error = (int)e;
  return GBMOE_CUDA_ERROR;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v) { return (v + kWsAlign - 1) / kWsAlign * kWsAlign; }

// carve consecutive 256-byte aligned pieces out of a workspace
struct Carver {
  uint8_t *base;
  size_t off = 0;
  explicit Carver(void *b) : base(static_cast<uint8_t *>(b)) {}
  void *take(size_t bytes) {
    void *p = base ? base + off : nullptr;
    off += round_up(bytes);
    return p;
  }
};

// e4m3 with one scale per row of each GEMM operand (per token or per tensor
// for the activations, per channel for the weights)
bool row_scaled(int dtype) {
  return dtype == GBMOE_FP8_E4M3_CHANNEL || dtype == GBMOE_FP8_E4M3_TENSOR;
}
bool is_fp8(int dtype) { return dtype == GBMOE_FP8_E4M3 || row_scaled(dtype); }
size_t elem_bytes(int dtype) { return is_fp8(dtype) ? 1 : 2; }
// fp32 scales per row of a (rows, cols) e4m3 operand: one per 128 columns,
// or one per row (row-scaled e4m3)
int scales_per_row(int dtype, int cols) { return row_scaled(dtype) ? 1 : cols / 128; }

// leading dimension of the group-major FP8 row scales of M*topk rows
int64_t scale_ld(size_t P) { return (int64_t)((P + 3) / 4 * 4); }

bool valid_dtype(int dtype) { return dtype == GBMOE_BF16 || is_fp8(dtype); }

struct ForwardWs {
  int32_t *ids, *counts, *offsets, *sorted, *inv, *chunk_hist;
  float *weights;
  void *A;
  float *As;
  void *H;
  float *Hs;
  uint16_t *Hb;     // row-scaled e4m3: H in bf16 before its quantisation
  uint32_t *amax;   // GBMOE_FP8_E4M3_TENSOR: the maxima of x and of H
  uint16_t *y_slot;
};
ForwardWs carve_forward(Carver &c, int M, int E, int N, int K, int topk, int dtype) {
  const size_t P = (size_t)M * topk;
  ForwardWs w;
  w.ids = static_cast<int32_t *>(c.take(P * 4));
  w.weights = static_cast<float *>(c.take(P * 4));
  w.counts = static_cast<int32_t *>(c.take((size_t)E * 4));
  w.offsets = static_cast<int32_t *>(c.take((size_t)(E + 1) * 4));
  w.sorted = static_cast<int32_t *>(c.take(P * 4));
  w.inv = static_cast<int32_t *>(c.take(P * 4));
  w.chunk_hist = static_cast<int32_t *>(c.take((size_t)align_num_chunks((int)P) * E * 4));
  const bool fp8 = is_fp8(dtype);
  const int sk = scales_per_row(dtype, K), sn = scales_per_row(dtype, N);
  w.A = c.take(P * (size_t)K * elem_bytes(dtype));
  w.As = fp8 ? static_cast<float *>(c.take((size_t)scale_ld(P) * sk * 4)) : nullptr;
  w.H = c.take(P * (size_t)N * elem_bytes(dtype));
  w.Hs = fp8 ? static_cast<float *>(c.take((size_t)scale_ld(P) * sn * 4)) : nullptr;
  w.Hb = row_scaled(dtype) ? static_cast<uint16_t *>(c.take(P * (size_t)N * 2)) : nullptr;
  w.amax = dtype == GBMOE_FP8_E4M3_TENSOR ? static_cast<uint32_t *>(c.take(2 * sizeof(uint32_t)))
                                         : nullptr;
  w.y_slot = static_cast<uint16_t *>(c.take(P * (size_t)K * 2));
  return w;
}

// BatchedExperts scratch: H (E*T, N) (bf16, or e4m3 with its group-major
// scales), and for e4m3 the activations' scales moved to the group-major
// layout the GEMM's scale loads read
struct BatchedWs {
  void *H;
  float *Hs;
  float *xs;
};
BatchedWs carve_batched(Carver &c, int T, int E, int N, int K, int dtype) {
  const size_t R = (size_t)E * T;
  BatchedWs w;
  w.H = c.take(R * (size_t)N * elem_bytes(dtype));
  const bool fp8 = dtype == GBMOE_FP8_E4M3;
  w.Hs = fp8 ? static_cast<float *>(c.take((size_t)scale_ld(R) * (N / 128) * 4)) : nullptr;
  w.xs = fp8 ? static_cast<float *>(c.take((size_t)scale_ld(R) * (K / 128) * 4)) : nullptr;
  return w;
}

// moe_shared_expert_forward: H (M, Ns), the down GEMM's operand.  Block
// e4m3 adds the codes of x, x's scales row-major (the quantiser's output)
// and group-major (the GEMM's operand), and H's group-major scales;
// per-channel e4m3 adds H's scale per row, H in bf16 before its quantisation,
// the codes of x and x's scale per row.
struct SharedWs {
  void *H;
  float *Hs;
  void *Hb;
  void *xq;
  float *xs_rows;
  float *xs;
};
SharedWs carve_shared(Carver &c, int M, int Ns, int K, int dtype) {
  SharedWs w{};
  w.H = c.take((size_t)M * Ns * elem_bytes(dtype));
  if (dtype == GBMOE_FP8_E4M3) {
    w.Hs = static_cast<float *>(c.take((size_t)scale_ld(M) * (Ns / 128) * 4));
    w.xq = c.take((size_t)M * K);
    w.xs_rows = static_cast<float *>(c.take((size_t)M * (K / 128) * 4));
    w.xs = static_cast<float *>(c.take((size_t)scale_ld(M) * (K / 128) * 4));
  } else if (dtype == GBMOE_FP8_E4M3_CHANNEL) {
    w.Hs = static_cast<float *>(c.take((size_t)M * 4));
    w.Hb = c.take((size_t)M * Ns * 2);
    w.xq = c.take((size_t)M * K);
    w.xs_rows = static_cast<float *>(c.take((size_t)M * 4));
  }
  return w;
}

EpWorkspace carve_ep(Carver &c, int G, int M, int E, int topk) {
  const size_t P = (size_t)G * M * topk;
  EpWorkspace w;
  w.ids_eff = static_cast<int32_t *>(c.take(P * 4));
  w.map = static_cast<int32_t *>(c.take((size_t)(E + 1) * 4));
  w.counts = static_cast<int32_t *>(c.take((size_t)E * 4));
  w.offsets = static_cast<int32_t *>(c.take((size_t)(E + 1) * 4));
  w.sorted = static_cast<int32_t *>(c.take(P * 4));
  w.inv = static_cast<int32_t *>(c.take(P * 4));
  w.chunk_hist = static_cast<int32_t *>(c.take((size_t)align_num_chunks((int)P) * E * 4));
  return w;
}

bool ep_shape_ok(int G, int M, int K, int E, int topk, int worst) {
  return G >= 1 && M >= 0 && K >= 8 && K % 8 == 0 && E >= 1 && E <= kMaxExperts &&
         E % G == 0 && topk >= 1 && topk <= kMaxTopk && topk <= E && worst >= 1 &&
         (size_t)G * M * topk <= (size_t)INT32_MAX && (size_t)E * worst <= (size_t)INT32_MAX;
}

// expert_map NULL: the routed ids are local ids (E_global == E); otherwise
// E_global routed experts map to E local ones
bool map_args_ok(int E_global, const int32_t *expert_map, int E) {
  if (E_global < 1) return false;
  return expert_map ? E_global <= (1 << 24) : E_global == E;
}

bool route_args_ok(int M, int E, int topk, int score_fn, const float *bias,
                   int n_groups, int topk_groups) {
  if (M < 0 || E < 1 || E > kMaxExperts || topk < 1 || topk > kMaxTopk || topk > E)
    return false;
  if (score_fn == GBMOE_SOFTMAX) return bias == nullptr;
  if (score_fn != GBMOE_SIGMOID) return false;
  if (n_groups > 1) {
    if (n_groups > 32 || E % n_groups != 0) return false;
    if (topk_groups < 1 || topk_groups > n_groups) return false;
    if (topk > topk_groups * (E / n_groups)) return false;
  }
  return true;
}

gbmoe_status_t gate_up_impl(const void *A, const float *A_scales,
                            const int32_t *offsets, int M, int topk, int E,
                            int N, int K, const void *w1, const float *w1_scales,
                            int dtype, int act, void *H, float *H_scales,
                            int32_t *err, int num_sms, cudaStream_t s) {
  GroupedGemmArgs a{};
  a.mode = kGateUp;
  a.act = act;
  a.fp8 = dtype == GBMOE_FP8_E4M3;
  a.fp8ch = row_scaled(dtype);
  a.offsets = offsets;
  a.E = E;
  a.N = N;
  a.K = K;
  a.A = A;
  a.a_rows = (int64_t)M * topk;
  a.A_scales = A_scales;
  a.scale_ld = scale_ld((size_t)M * topk);
  a.B = w1;
  a.B_scales = w1_scales;
  a.out = H;
  a.out_scales = H_scales;
  a.err = err;
  return from_cuda(launch_grouped_gemm(a, num_sms, s));
}

gbmoe_status_t permute_impl(const void *x, const float *x_scales,
                            const float *row_weights, const int32_t *sorted,
                            const int32_t *offsets, int M, int topk, int E, int K,
                            int dtype, void *A, float *A_scales, int num_sms,
                            cudaStream_t s) {
  const bool fp8 = is_fp8(dtype);
  return from_cuda(launch_gather_rows(x, fp8 ? x_scales : nullptr,
                                      fp8 ? nullptr : row_weights,
                                      (int)(K * elem_bytes(dtype)), scales_per_row(dtype, K),
                                      sorted,
                                      offsets + E, M * topk, topk, A,
                                      fp8 ? A_scales : nullptr,
                                      scale_ld((size_t)M * topk), num_sms, s));
}

gbmoe_status_t down_impl(const void *H, const float *H_scales,
                         const int32_t *sorted, const int32_t *offsets,
                         const float *topk_weights, int M, int topk, int E,
                         int N, int K, const void *w2, const float *w2_scales,
                         int dtype, uint16_t *y_slot, int32_t *err, int num_sms,
                         cudaStream_t s) {
  GroupedGemmArgs a{};
  a.mode = kDown;
  a.fp8 = dtype == GBMOE_FP8_E4M3;
  a.fp8ch = row_scaled(dtype);
  a.offsets = offsets;
  a.E = E;
  a.N = N;
  a.K = K;
  a.A = H;
  a.a_rows = (int64_t)M * topk;
  a.A_scales = H_scales;
  a.scale_ld = scale_ld((size_t)M * topk);
  a.B = w2;
  a.B_scales = w2_scales;
  a.out = y_slot;
  a.sorted_pair_ids = sorted;
  a.topk_weights = topk_weights;
  a.err = err;
  return from_cuda(launch_grouped_gemm(a, num_sms, s));
}

// K and N of the block-scaled e4m3 GEMMs: the weight-block scales of a tile
// (two rows of K/128 or N/128 values) are staged in shared memory, 128 each
constexpr int kMaxFp8BlockK = 16384;

bool gemm_shape_ok(int M, int topk, int E, int N, int K, int dtype) {
  return M >= 0 && topk >= 1 && topk <= kMaxTopk && E >= 1 && E <= kMaxExperts &&
         N >= 128 && K >= 128 && N % 128 == 0 && K % 128 == 0 && valid_dtype(dtype) &&
         (dtype != GBMOE_FP8_E4M3 || (K <= kMaxFp8BlockK && N <= kMaxFp8BlockK)) &&
         (size_t)M * topk <= (size_t)INT32_MAX && (size_t)E * 2 * N <= (size_t)INT32_MAX &&
         (size_t)E * K <= (size_t)INT32_MAX;
}

}  // namespace

gbmoe_status_t status_from_cuda(cudaError_t e) { return from_cuda(e); }

}  // namespace gbmoe

using namespace gbmoe;

extern "C" {

const char *gbmoe_status_string(gbmoe_status_t status) {
  switch (status) {
    case GBMOE_OK: return "ok";
    case GBMOE_INVALID_ARG: return "invalid argument";
    case GBMOE_UNSUPPORTED: return "unsupported dtype or device";
    case GBMOE_CUDA_ERROR: return "CUDA launch error";
  }
  return "unknown status";
}

int gbmoe_last_cuda_error(void) { return g_last_cuda_error; }

size_t moe_workspace_size(int which, int M_or_T, int E, int N, int K, int topk,
                          int dtype) {
  if (M_or_T < 0 || E < 1 || E > kMaxExperts) return 0;
  Carver c(nullptr);
  switch (which) {
    case GBMOE_WS_ALIGN: {
      if (topk < 1) return 0;
      const size_t P = (size_t)M_or_T * topk;
      c.take((size_t)align_num_chunks((int)P) * E * 4);
      return c.off > 0 ? c.off : kWsAlign;
    }
    case GBMOE_WS_BATCHED:
      if (!gemm_shape_ok(M_or_T, 1, E, N, K, dtype) ||
          (dtype != GBMOE_BF16 && dtype != GBMOE_FP8_E4M3) || (size_t)E * M_or_T > (size_t)INT32_MAX)
        return 0;
      carve_batched(c, M_or_T, E, N, K, dtype);
      return c.off > 0 ? c.off : kWsAlign;
    case GBMOE_WS_FORWARD:
      if (!gemm_shape_ok(M_or_T, topk, E, N, K, dtype)) return 0;
      carve_forward(c, M_or_T, E, N, K, topk, dtype);
      return c.off;
    case GBMOE_WS_EP_DISPATCH:
      // M_or_T: tokens per shard (M), E: all routed experts, N: the number of
      // shards G
      if (topk < 1 || N < 1 || E % N != 0 || (size_t)N * M_or_T * topk > (size_t)INT32_MAX)
        return 0;
      carve_ep(c, N, M_or_T, E, topk);
      return c.off;
    case GBMOE_WS_SHARED:
      if (dtype != GBMOE_BF16 && dtype != GBMOE_FP8_E4M3 && dtype != GBMOE_FP8_E4M3_CHANNEL)
        return 0;
      if (!gemm_shape_ok(M_or_T, 1, 1, N, K, dtype)) return 0;
      carve_shared(c, M_or_T, N, K, dtype);
      return c.off > 0 ? c.off : kWsAlign;
  }
  return 0;
}

gbmoe_status_t moe_topk_route(const float *logits, const float *bias, int M,
                              int E, int topk, int score_fn, int n_groups,
                              int topk_groups, int renormalize,
                              int32_t *topk_ids, float *topk_weights,
                              int32_t *err_word, gbmoe_stream_t stream) {
  (void)err_word;
  if (!route_args_ok(M, E, topk, score_fn, bias, n_groups, topk_groups))
    return GBMOE_INVALID_ARG;
  if (M > 0 && (!logits || !topk_ids || !topk_weights)) return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (M == 0) return GBMOE_OK;
  return from_cuda(launch_route(logits, bias, M, E, topk, score_fn,
                                n_groups < 1 ? 1 : n_groups, topk_groups,
                                renormalize, topk_ids, topk_weights,
                                (cudaStream_t)stream));
}

gbmoe_status_t moe_count_expert_tokens(const int32_t *topk_ids, int M,
                                       int topk, int E_global,
                                       const int32_t *expert_map, int E,
                                       int32_t *counts, int32_t *err_word,
                                       gbmoe_stream_t stream) {
  if (M < 0 || topk < 1 || E < 1 || E > kMaxExperts || !counts) return GBMOE_INVALID_ARG;
  if (!map_args_ok(E_global, expert_map, E)) return GBMOE_INVALID_ARG;
  if (M > 0 && !topk_ids) return GBMOE_INVALID_ARG;
  if ((size_t)M * topk > (size_t)INT32_MAX) return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (M == 0)
    return from_cuda(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, (cudaStream_t)stream));
  return from_cuda(launch_count(topk_ids, M * topk, E_global, expert_map, E, counts,
                                err_word, sms, (cudaStream_t)stream));
}

gbmoe_status_t moe_align_permute(const int32_t *topk_ids, int M, int topk,
                                 int E_global, const int32_t *expert_map, int E,
                                 int32_t *counts, int32_t *offsets,
                                 int32_t *sorted_pair_ids, int32_t *inv,
                                 void *ws, size_t ws_bytes, int32_t *err_word,
                                 gbmoe_stream_t stream) {
  if (M < 0 || topk < 1 || E < 1 || E > kMaxExperts || !offsets) return GBMOE_INVALID_ARG;
  if (!map_args_ok(E_global, expert_map, E)) return GBMOE_INVALID_ARG;
  if ((size_t)M * topk > (size_t)INT32_MAX) return GBMOE_INVALID_ARG;
  if (M > 0 && (!topk_ids || !sorted_pair_ids || !inv || !ws)) return GBMOE_INVALID_ARG;
  if (ws_bytes < moe_workspace_size(GBMOE_WS_ALIGN, M, E, 0, 0, topk, 0)) return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  return from_cuda(launch_align(topk_ids, M * topk, E_global, expert_map, E, counts, offsets,
                                sorted_pair_ids, inv, static_cast<int32_t *>(ws),
                                err_word, (cudaStream_t)stream));
}

gbmoe_status_t moe_quant_fp8_group(const uint16_t *x, const float *row_weights,
                                   int M, int K, int group, uint8_t *q,
                                   float *scales, gbmoe_stream_t stream) {
  if (M < 0 || K < 128 || K % 128 != 0 || (group != 128 && group != K))
    return GBMOE_INVALID_ARG;
  if (M > 0 && (!x || !q || !scales || !aligned16(x) || !aligned16(q)))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (M == 0) return GBMOE_OK;
  if (group == K && K != 128)  // one group per row
    return from_cuda(
        launch_quant_row(x, row_weights, M, K, q, scales, sms, (cudaStream_t)stream));
  return from_cuda(
      launch_quant_group(x, row_weights, M, K, q, scales, sms, (cudaStream_t)stream));
}

gbmoe_status_t moe_quant_fp8_group_permute(const uint16_t *x, const float *row_weights,
                                           int M, int K, const int32_t *inv, int topk,
                                           uint8_t *A, float *A_scales, gbmoe_stream_t stream) {
  if (M < 0 || K < 128 || K % 128 != 0 || topk < 1 || topk > kMaxTopk) return GBMOE_INVALID_ARG;
  if (row_weights && topk != 1) return GBMOE_INVALID_ARG;
  if ((size_t)M * topk > (size_t)INT32_MAX) return GBMOE_INVALID_ARG;
  if (M > 0 && (!x || !inv || !A || !A_scales || !aligned16(x) || !aligned16(A) ||
                (reinterpret_cast<uintptr_t>(A_scales) & 3u)))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  return from_cuda(launch_quant_group_scatter(x, row_weights, M, K, inv, topk, A, A_scales,
                                              scale_ld((size_t)M * topk), sms,
                                              (cudaStream_t)stream));
}

gbmoe_status_t moe_quant_fp8_row_permute(const uint16_t *x, const float *row_weights,
                                         int M, int K, const int32_t *inv, int topk,
                                         uint8_t *A, float *A_scales, gbmoe_stream_t stream) {
  if (M < 0 || K < 128 || K % 128 != 0 || topk < 1 || topk > kMaxTopk) return GBMOE_INVALID_ARG;
  if (row_weights && topk != 1) return GBMOE_INVALID_ARG;
  if ((size_t)M * topk > (size_t)INT32_MAX) return GBMOE_INVALID_ARG;
  if (M > 0 && (!x || !inv || !A || !A_scales || !aligned16(x) || !aligned16(A) ||
                (reinterpret_cast<uintptr_t>(A_scales) & 3u)))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  return from_cuda(launch_quant_row_scatter(x, row_weights, M, K, inv, topk, A, A_scales, sms,
                                            (cudaStream_t)stream));
}

gbmoe_status_t moe_quant_fp8_tensor_permute(const uint16_t *x, const float *row_weights,
                                            int M, int K, const int32_t *inv, int topk,
                                            const float *scale, uint8_t *A, float *A_scales,
                                            uint32_t *amax_ws, gbmoe_stream_t stream) {
  if (M < 0 || K < 128 || K % 128 != 0 || topk < 1 || topk > kMaxTopk) return GBMOE_INVALID_ARG;
  if (row_weights && topk != 1) return GBMOE_INVALID_ARG;
  if ((size_t)M * topk > (size_t)INT32_MAX) return GBMOE_INVALID_ARG;
  if (M > 0 && (!x || !inv || !A || !A_scales || !aligned16(x) || !aligned16(A) ||
                (reinterpret_cast<uintptr_t>(A_scales) & 3u) ||
                (reinterpret_cast<uintptr_t>(scale) & 3u) ||
                (!scale && (!amax_ws || (reinterpret_cast<uintptr_t>(amax_ws) & 3u)))))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  return from_cuda(launch_quant_tensor_scatter(x, row_weights, M, K, inv, topk, A, A_scales,
                                               amax_ws, scale, sms, (cudaStream_t)stream));
}

gbmoe_status_t moe_quant_fp8_tensor(const uint16_t *x, const float *row_weights,
                                    int M, int K, const int32_t *n_rows,
                                    uint8_t *q, float *row_scales,
                                    uint32_t *amax_ws, gbmoe_stream_t stream) {
  if (M < 0 || K < 128 || K % 128 != 0) return GBMOE_INVALID_ARG;
  if (M > 0 && (!x || !q || !row_scales || !amax_ws || !aligned16(x) || !aligned16(q) ||
                reinterpret_cast<uintptr_t>(amax_ws) % 4 != 0))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (M == 0) return GBMOE_OK;
  return from_cuda(launch_quant_tensor(x, row_weights, M, K, n_rows, q, row_scales, amax_ws,
                                       nullptr, sms, (cudaStream_t)stream));
}

gbmoe_status_t moe_quant_fp8_tensor_static(const uint16_t *x, const float *row_weights,
                                           int M, int K, const int32_t *n_rows,
                                           const float *scale, uint8_t *q, float *row_scales,
                                           gbmoe_stream_t stream) {
  if (M < 0 || K < 128 || K % 128 != 0) return GBMOE_INVALID_ARG;
  if (M > 0 && (!x || !q || !row_scales || !scale || !aligned16(x) || !aligned16(q) ||
                reinterpret_cast<uintptr_t>(scale) % 4 != 0))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (M == 0) return GBMOE_OK;
  return from_cuda(launch_quant_tensor(x, row_weights, M, K, n_rows, q, row_scales, nullptr,
                                       scale, sms, (cudaStream_t)stream));
}

gbmoe_status_t moe_quant_fp8_block(const uint16_t *w, int64_t R, int C,
                                   int block, uint8_t *q, float *scales,
                                   gbmoe_stream_t stream) {
  if (R < 0 || C < 128 || R % 128 != 0 || C % 128 != 0 || block != 128)
    return GBMOE_INVALID_ARG;
  if ((R / 128) * (C / 128) > (int64_t)INT32_MAX) return GBMOE_INVALID_ARG;
  if (R > 0 && (!w || !q || !scales || !aligned16(w) || !aligned16(q)))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (R == 0) return GBMOE_OK;
  return from_cuda(launch_quant_block(w, R, C, q, scales, (cudaStream_t)stream));
}

gbmoe_status_t moe_permute_rows(const void *x, const float *x_scales,
                                const float *row_weights,
                                const int32_t *sorted_pair_ids,
                                const int32_t *offsets, int M, int topk, int E,
                                int K, int dtype, void *A, float *A_scales,
                                gbmoe_stream_t stream) {
  if (!valid_dtype(dtype)) return GBMOE_UNSUPPORTED;
  if (M < 0 || topk < 1 || topk > kMaxTopk || E < 1 || E > kMaxExperts || K < 128 ||
      K % 128 != 0 || (size_t)M * topk > (size_t)INT32_MAX)
    return GBMOE_INVALID_ARG;
  const bool fp8 = is_fp8(dtype);
  if (M > 0) {
    if (!x || !sorted_pair_ids || !offsets || !A || !aligned16(x) || !aligned16(A))
      return GBMOE_INVALID_ARG;
    if (fp8 && (!x_scales || !A_scales)) return GBMOE_INVALID_ARG;
  }
  // FP8 rows take their router weight in moe_quant_fp8_group, before the codes
  if (fp8 && row_weights) return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  return permute_impl(x, x_scales, row_weights, sorted_pair_ids, offsets, M, topk, E, K,
                      dtype, A, A_scales, sms, (cudaStream_t)stream);
}

static gbmoe_status_t gate_up_entry(
    const void *A, const float *A_scales, const int32_t *offsets, int M,
    int topk, int E, int N, int K, const void *w1, const float *w1_scales,
    int dtype, int act, void *H, float *H_scales, int32_t *err_word,
    gbmoe_stream_t stream) {
  if (!valid_dtype(dtype)) return GBMOE_UNSUPPORTED;
  if (!gemm_shape_ok(M, topk, E, N, K, dtype)) return GBMOE_INVALID_ARG;
  const bool fp8 = dtype == GBMOE_FP8_E4M3;
  const bool fp8ch = row_scaled(dtype);
  if (M > 0) {
    if (!A || !offsets || !w1 || !H) return GBMOE_INVALID_ARG;
    if (fp8 && (!A_scales || !w1_scales || !H_scales)) return GBMOE_INVALID_ARG;
    if (fp8ch && (!A_scales || !w1_scales || !aligned16(w1_scales))) return GBMOE_INVALID_ARG;
    if (!aligned16(A) || !aligned16(w1) || !aligned16(H)) return GBMOE_INVALID_ARG;
  }
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  return gate_up_impl(A, A_scales, offsets, M, topk, E, N, K, w1, w1_scales, dtype, act, H,
                      H_scales, err_word, sms, (cudaStream_t)stream);
}

gbmoe_status_t moe_grouped_gemm_gate_up_silu(
    const void *A, const float *A_scales, const int32_t *offsets, int M,
    int topk, int E, int N, int K, const void *w1, const float *w1_scales,
    int dtype, void *H, float *H_scales, int32_t *err_word,
    gbmoe_stream_t stream) {
  return gate_up_entry(A, A_scales, offsets, M, topk, E, N, K, w1, w1_scales, dtype,
                       GBMOE_ACT_SILU, H, H_scales, err_word, stream);
}

gbmoe_status_t moe_grouped_gemm_gate_up_gelu(
    const void *A, const float *A_scales, const int32_t *offsets, int M,
    int topk, int E, int N, int K, const void *w1, const float *w1_scales,
    int dtype, void *H, float *H_scales, int32_t *err_word,
    gbmoe_stream_t stream) {
  return gate_up_entry(A, A_scales, offsets, M, topk, E, N, K, w1, w1_scales, dtype,
                       GBMOE_ACT_GELU, H, H_scales, err_word, stream);
}

gbmoe_status_t moe_grouped_gemm_down(
    const void *H, const float *H_scales, const int32_t *sorted_pair_ids,
    const int32_t *offsets, const float *topk_weights, int M, int topk, int E,
    int N, int K, const void *w2, const float *w2_scales, int dtype,
    uint16_t *y_slot, int32_t *err_word, gbmoe_stream_t stream) {
  if (!valid_dtype(dtype)) return GBMOE_UNSUPPORTED;
  if (!gemm_shape_ok(M, topk, E, N, K, dtype)) return GBMOE_INVALID_ARG;
  if (M == 0) {
    int sms;
    return device_info(&sms);
  }
  const bool fp8 = is_fp8(dtype);
  if (!H || !sorted_pair_ids || !offsets || !w2 || !y_slot) return GBMOE_INVALID_ARG;
  if (fp8 && (!H_scales || !w2_scales)) return GBMOE_INVALID_ARG;
  if (row_scaled(dtype) && !aligned16(w2_scales)) return GBMOE_INVALID_ARG;
  if (!aligned16(H) || !aligned16(w2) || !aligned16(y_slot)) return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  return down_impl(H, H_scales, sorted_pair_ids, offsets, topk_weights, M, topk, E, N,
                   K, w2, w2_scales, dtype, y_slot, err_word, sms,
                   (cudaStream_t)stream);
}

gbmoe_status_t moe_ep_dispatch(const void *x, const float *x_scales,
                               const int32_t *num_tokens, const int32_t *topk_ids,
                               int G, int M, int K, int E, int topk, int worst_tokens,
                               int dtype, void *recv_x, float *recv_scales,
                               int32_t *recv_counts, int32_t *recv_pos, void *ws,
                               size_t ws_bytes, int32_t *err_word, gbmoe_stream_t stream) {
  if (dtype != GBMOE_BF16 && dtype != GBMOE_FP8_E4M3) return GBMOE_UNSUPPORTED;
  const bool fp8 = dtype == GBMOE_FP8_E4M3;
  if (!ep_shape_ok(G, M, K, E, topk, worst_tokens) || (fp8 && K % 128 != 0))
    return GBMOE_INVALID_ARG;
  if (M > 0) {
    if (!x || !num_tokens || !topk_ids || !recv_x || !recv_counts || !recv_pos || !ws)
      return GBMOE_INVALID_ARG;
    if (fp8 && (!x_scales || !recv_scales || (reinterpret_cast<uintptr_t>(x_scales) & 3u) ||
                (reinterpret_cast<uintptr_t>(recv_scales) & 3u)))
      return GBMOE_INVALID_ARG;
    if (!aligned16(x) || !aligned16(recv_x) || !aligned16(ws)) return GBMOE_INVALID_ARG;
    if (ws_bytes < moe_workspace_size(GBMOE_WS_EP_DISPATCH, M, E, G, K, topk, 0))
      return GBMOE_INVALID_ARG;
  }
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (M == 0)  // nothing routed: every expert receives no row
    return from_cuda(cudaMemsetAsync(recv_counts, 0, (size_t)E * 4, s));
  Carver c(ws);
  EpWorkspace w = carve_ep(c, G, M, E, topk);
  return from_cuda(launch_ep_dispatch(x, fp8 ? x_scales : nullptr, num_tokens, topk_ids, G, M, K,
                                      (int)elem_bytes(dtype) * K, E, topk, worst_tokens, recv_x,
                                      fp8 ? recv_scales : nullptr, recv_counts, recv_pos, w,
                                      err_word, sms, s));
}

gbmoe_status_t moe_ep_combine(const uint16_t *recv_y, const int32_t *topk_ids,
                              const int32_t *recv_pos, const float *topk_weights,
                              const int32_t *num_tokens, int G, int M, int K, int E,
                              int topk, int worst_tokens, uint16_t *out,
                              gbmoe_stream_t stream) {
  if (!ep_shape_ok(G, M, K, E, topk, worst_tokens)) return GBMOE_INVALID_ARG;
  if (M > 0) {
    if (!recv_y || !topk_ids || !recv_pos || !topk_weights || !num_tokens || !out)
      return GBMOE_INVALID_ARG;
    if (!aligned16(recv_y) || !aligned16(out)) return GBMOE_INVALID_ARG;
  }
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  return from_cuda(launch_ep_combine(recv_y, topk_ids, recv_pos, topk_weights, num_tokens, G, M,
                                     K, E, topk, worst_tokens, out, sms, (cudaStream_t)stream));
}

gbmoe_status_t moe_unpermute_weighted_reduce(const uint16_t *y_slot,
                                             const int32_t *inv, int M,
                                             int topk, int K, uint16_t *out,
                                             gbmoe_stream_t stream) {
  if (M < 0 || topk < 1 || topk > kMaxTopk || K < 8 || K % 8 != 0) return GBMOE_INVALID_ARG;
  if (M > 0 && (!y_slot || !out || !aligned16(y_slot) || !aligned16(out)))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (M == 0) return GBMOE_OK;
  return from_cuda(launch_reduce(y_slot, inv, M, topk, K, out, sms, (cudaStream_t)stream));
}

gbmoe_status_t moe_batched_masked_experts(
    const void *x_b, const float *x_b_scales,
    const int32_t *expert_num_tokens, int E, int T, int N, int K,
    const void *w1, const float *w1_scales, const void *w2,
    const float *w2_scales, int dtype, int activation, uint16_t *y_b, void *ws,
    size_t ws_bytes, int32_t *err_word, gbmoe_stream_t stream) {
  if (activation != GBMOE_ACT_SILU && activation != GBMOE_ACT_GELU) return GBMOE_INVALID_ARG;
  if (dtype != GBMOE_BF16 && dtype != GBMOE_FP8_E4M3) return GBMOE_UNSUPPORTED;
  const bool fp8 = dtype == GBMOE_FP8_E4M3;
  if (!gemm_shape_ok(T, 1, E, N, K, dtype)) return GBMOE_INVALID_ARG;
  if ((size_t)E * T > (size_t)INT32_MAX) return GBMOE_INVALID_ARG;
  if (T == 0) {
    int sms;
    return device_info(&sms);
  }
  if (!x_b || !expert_num_tokens || !w1 || !w2 || !y_b || !ws) return GBMOE_INVALID_ARG;
  if (fp8 && (!x_b_scales || !w1_scales || !w2_scales)) return GBMOE_INVALID_ARG;
  if (fp8 && (reinterpret_cast<uintptr_t>(x_b_scales) & 3u)) return GBMOE_INVALID_ARG;
  if (!aligned16(x_b) || !aligned16(w1) || !aligned16(w2) || !aligned16(y_b) || !aligned16(ws))
    return GBMOE_INVALID_ARG;
  if (ws_bytes < moe_workspace_size(GBMOE_WS_BATCHED, T, E, N, K, 1, dtype))
    return GBMOE_INVALID_ARG;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  Carver c(ws);
  const BatchedWs w = carve_batched(c, T, E, N, K, dtype);
  const int64_t R = (int64_t)E * T;
  GroupedGemmArgs a{};
  a.mode = kGateUp;
  a.fp8 = fp8;
  a.act = activation;
  a.counts = expert_num_tokens;
  a.E = E;
  a.T = T;
  a.N = N;
  a.K = K;
  a.A = x_b;
  a.a_rows = R;
  a.B = w1;
  a.out = w.H;
  a.err = err_word;
  cudaError_t ce;
  if (fp8) {
    // the caller's (E*T, K/128) row-major scales -> (K/128, ld) group-major,
    // for the runs of rows that hold valid tokens (the GEMM stores no other)
    ce = launch_scales_group_major(x_b_scales, R, K / 128, w.xs, scale_ld((size_t)R), sms, s,
                                   expert_num_tokens, T);
    if (ce != cudaSuccess) return from_cuda(ce);
    a.A_scales = w.xs;
    a.scale_ld = scale_ld((size_t)R);
    a.B_scales = w1_scales;
    a.out_scales = w.Hs;
  }
  ce = launch_grouped_gemm(a, sms, s);
  if (ce != cudaSuccess) return from_cuda(ce);
  a.mode = kDown;
  a.A = w.H;
  a.A_scales = w.Hs;
  a.B = w2;
  a.B_scales = w2_scales;
  a.out_scales = nullptr;
  a.out = y_b;
  return from_cuda(launch_grouped_gemm(a, sms, s));
}

// every argument check of moe_forward (no launch, no device query)
static gbmoe_status_t forward_validate(const uint16_t *x, const float *logits,
                                       const float *bias, int M, int K, int N,
                                       int E_global, const int32_t *expert_map, int E,
                                       int topk, int score_fn, int n_groups,
                                       int topk_groups, int apply_router_weight_on_input,
                                       int activation, int dtype, const void *w1,
                                       const float *w1_scales, const void *w2,
                                       const float *w2_scales, const float *a1_scale,
                                       const float *a2_scale, const uint16_t *out,
                                       const void *ws, size_t ws_bytes) {
  if (!valid_dtype(dtype)) return GBMOE_UNSUPPORTED;
  // static activation scales: per-tensor e4m3 only, each a device fp32
  if ((a1_scale || a2_scale) && dtype != GBMOE_FP8_E4M3_TENSOR) return GBMOE_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a1_scale) & 3u) || (reinterpret_cast<uintptr_t>(a2_scale) & 3u))
    return GBMOE_INVALID_ARG;
  if (!gemm_shape_ok(M, topk, E, N, K, dtype)) return GBMOE_INVALID_ARG;
  if (!map_args_ok(E_global, expert_map, E)) return GBMOE_INVALID_ARG;
  if (!route_args_ok(M, E_global, topk, score_fn, bias, n_groups, topk_groups))
    return GBMOE_INVALID_ARG;
  if (apply_router_weight_on_input && topk != 1) return GBMOE_INVALID_ARG;
  if (activation != GBMOE_ACT_SILU && activation != GBMOE_ACT_GELU) return GBMOE_INVALID_ARG;
  const bool fp8 = is_fp8(dtype);
  if (M > 0) {
    if (!x || !logits || !w1 || !w2 || !out || !ws) return GBMOE_INVALID_ARG;
    if (fp8 && (!w1_scales || !w2_scales)) return GBMOE_INVALID_ARG;
    if (row_scaled(dtype) && (!aligned16(w1_scales) || !aligned16(w2_scales)))
      return GBMOE_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w1) || !aligned16(w2) || !aligned16(out) || !aligned16(ws))
      return GBMOE_INVALID_ARG;
    if (ws_bytes < moe_workspace_size(GBMOE_WS_FORWARD, M, E, N, K, topk, dtype))
      return GBMOE_INVALID_ARG;
  }
  return GBMOE_OK;
}

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
                           int32_t *err_word, gbmoe_stream_t stream) {
  gbmoe_status_t vst = forward_validate(x, logits, bias, M, K, N, E_global, expert_map, E,
                                        topk, score_fn, n_groups, topk_groups,
                                        apply_router_weight_on_input, activation, dtype, w1,
                                        w1_scales, w2, w2_scales, a1_scale, a2_scale, out, ws,
                                        ws_bytes);
  if (vst != GBMOE_OK) return vst;
  const bool fp8 = is_fp8(dtype);
  const bool fp8ch = row_scaled(dtype);
  const bool fp8t = dtype == GBMOE_FP8_E4M3_TENSOR;
  int sms;
  gbmoe_status_t st = device_info(&sms);
  if (st != GBMOE_OK) return st;
  if (M == 0) return GBMOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  Carver c(ws);
  ForwardWs w = carve_forward(c, M, E, N, K, topk, dtype);
  int32_t *ids = topk_ids ? topk_ids : w.ids;
  float *wts = topk_weights ? topk_weights : w.weights;
  const int P = M * topk;
  cudaError_t ce = launch_route(logits, bias, M, E_global, topk, score_fn,
                                n_groups < 1 ? 1 : n_groups, topk_groups, renormalize,
                                ids, wts, s);
  if (ce != cudaSuccess) return from_cuda(ce);
  ce = launch_align(ids, P, E_global, expert_map, E, w.counts, w.offsets, w.sorted, w.inv,
                    w.chunk_hist, err_word, s);
  if (ce != cudaSuccess) return from_cuda(ce);
  // apply_router_weight_on_input (top-1): the weight scales the activations
  // (before the FP8 codes are chosen) and not the expert output
  const float *in_w = apply_router_weight_on_input ? wts : nullptr;
  if (fp8 && !fp8t && !fp8ch) {
    // 1 x 128 groups: the codes and scales go straight to the permuted rows
    ce = launch_quant_group_scatter(x, in_w, M, K, w.inv, topk, static_cast<uint8_t *>(w.A),
                                    w.As, scale_ld((size_t)P), sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
  } else if (fp8ch && !fp8t) {
    // one scale per token: likewise, the row's codes and its scale to every
    // permuted row of the token's pairs
    ce = launch_quant_row_scatter(x, in_w, M, K, w.inv, topk, static_cast<uint8_t *>(w.A), w.As,
                                  sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
  } else if (fp8t) {
    // one scale for the tensor (its maximum, or a1_scale): the codes pass
    // writes the permuted rows
    ce = launch_quant_tensor_scatter(x, in_w, M, K, w.inv, topk, static_cast<uint8_t *>(w.A),
                                     w.As, w.amax, a1_scale, sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
  } else {  // bf16: the rows gathered (times the weight on input)
    st = permute_impl(x, nullptr, in_w, w.sorted, w.offsets, M, topk, E, K, dtype, w.A, w.As,
                      sms, s);
    if (st != GBMOE_OK) return st;
  }
  // per-token (per-tensor) scales span a whole row (all computed rows) of
  // H: it is written in bf16 and quantised before the second GEMM
  st = gate_up_impl(w.A, w.As, w.offsets, M, topk, E, N, K, w1, w1_scales, dtype, activation,
                    fp8ch ? static_cast<void *>(w.Hb) : w.H, w.Hs, err_word, sms, s);
  if (st != GBMOE_OK) return st;
  if (fp8t) {  // rows at and beyond offsets[E] (pairs not computed here) do not count
    ce = launch_quant_tensor(w.Hb, nullptr, P, N, w.offsets + E, static_cast<uint8_t *>(w.H),
                             w.Hs, w.amax + 1, a2_scale, sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
  } else if (fp8ch) {
    ce = launch_quant_row(w.Hb, nullptr, P, N, static_cast<uint8_t *>(w.H), w.Hs, sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
  }
  st = down_impl(w.H, w.Hs, w.sorted, w.offsets, in_w ? nullptr : wts, M, topk, E, N, K, w2,
                 w2_scales, dtype, w.y_slot, err_word, sms, s);
  if (st != GBMOE_OK) return st;
  return from_cuda(launch_reduce(w.y_slot, w.inv, M, topk, K, out, sms, s));
}

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
                                   int32_t *err_word, gbmoe_stream_t stream) {
  if (chunk_size < 1) return GBMOE_INVALID_ARG;
  const int CS = M < chunk_size ? M : chunk_size;
  // validate once with the chunk's size (the workspace is sized for it)
  gbmoe_status_t st = forward_validate(x, logits, bias, CS, K, N, E_global, expert_map, E,
                                       topk, score_fn, n_groups, topk_groups,
                                       apply_router_weight_on_input, activation, dtype, w1,
                                       w1_scales, w2, w2_scales, a1_scale, a2_scale, out, ws,
                                       ws_bytes);
  if (st != GBMOE_OK) return st;
  if (M < 0) return GBMOE_INVALID_ARG;
  for (int t0 = 0; t0 < M; t0 += CS) {
    const int m = M - t0 < CS ? M - t0 : CS;
    st = moe_forward(x + (size_t)t0 * K, logits + (size_t)t0 * E_global, bias, m, K, N,
                     E_global, expert_map, E, topk, score_fn, n_groups, topk_groups,
                     renormalize, apply_router_weight_on_input, activation, dtype, w1,
                     w1_scales, w2, w2_scales, a1_scale, a2_scale, out + (size_t)t0 * K,
                     topk_ids ? topk_ids + (size_t)t0 * topk : nullptr,
                     topk_weights ? topk_weights + (size_t)t0 * topk : nullptr, ws, ws_bytes,
                     err_word, stream);
    if (st != GBMOE_OK) return st;
  }
  return GBMOE_OK;
}

// every argument check of moe_shared_expert_forward (no launch, no device query)
static gbmoe_status_t shared_validate(const uint16_t *x, int M, int K, int Ns, const void *w1s,
                                      const float *w1s_scales, const void *w2s,
                                      const float *w2s_scales, int dtype, int activation,
                                      const uint16_t *out_shared, const void *ws,
                                      size_t ws_bytes) {
  if (dtype != GBMOE_BF16 && dtype != GBMOE_FP8_E4M3 && dtype != GBMOE_FP8_E4M3_CHANNEL)
    return GBMOE_UNSUPPORTED;
  if (!gemm_shape_ok(M, 1, 1, Ns, K, dtype)) return GBMOE_INVALID_ARG;
  if (activation != GBMOE_ACT_SILU && activation != GBMOE_ACT_GELU) return GBMOE_INVALID_ARG;
  if (M > 0) {
    if (!x || !w1s || !w2s || !out_shared || !ws) return GBMOE_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w1s) || !aligned16(w2s) || !aligned16(out_shared) ||
        !aligned16(ws))
      return GBMOE_INVALID_ARG;
    if (dtype == GBMOE_FP8_E4M3 &&
        (!w1s_scales || !w2s_scales || (reinterpret_cast<uintptr_t>(w1s_scales) & 3u) ||
         (reinterpret_cast<uintptr_t>(w2s_scales) & 3u)))
      return GBMOE_INVALID_ARG;
    // per-channel weight scales are read 16 bytes at a time
    if (dtype == GBMOE_FP8_E4M3_CHANNEL &&
        (!w1s_scales || !w2s_scales || !aligned16(w1s_scales) || !aligned16(w2s_scales)))
      return GBMOE_INVALID_ARG;
    if (ws_bytes < moe_workspace_size(GBMOE_WS_SHARED, M, 1, Ns, K, 1, dtype))
      return GBMOE_INVALID_ARG;
  }
  return GBMOE_OK;
}

gbmoe_status_t moe_shared_expert_forward(const uint16_t *x, int M, int K, int Ns,
                                         const void *w1s, const float *w1s_scales,
                                         const void *w2s, const float *w2s_scales,
                                         int dtype, int activation, uint16_t *out_shared,
                                         void *ws, size_t ws_bytes, int32_t *err_word,
                                         gbmoe_stream_t stream) {
  gbmoe_status_t st = shared_validate(x, M, K, Ns, w1s, w1s_scales, w2s, w2s_scales, dtype,
                                      activation, out_shared, ws, ws_bytes);
  if (st != GBMOE_OK) return st;
  int sms;
  st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const bool fp8 = dtype == GBMOE_FP8_E4M3;
  const bool fp8ch = dtype == GBMOE_FP8_E4M3_CHANNEL;
  Carver c(ws);
  const SharedWs w = carve_shared(c, M, Ns, K, dtype);
  // one expert owning all M rows ("dense": neither offsets nor counts)
  GroupedGemmArgs a{};
  a.mode = kGateUp;
  a.fp8 = fp8;
  a.act = activation;
  a.E = 1;
  a.T = M;
  a.N = Ns;
  a.K = K;
  a.A = x;
  a.a_rows = M;
  a.B = w1s;
  a.out = w.H;
  a.err = err_word;
  cudaError_t ce;
  if (fp8ch) {
    // one scale per token; h in bf16, then one scale per row of H
    ce = launch_quant_row(x, nullptr, M, K, static_cast<uint8_t *>(w.xq), w.xs_rows, sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
    a.fp8ch = true;
    a.A = w.xq;
    a.A_scales = w.xs_rows;
    a.scale_ld = scale_ld((size_t)M);
    a.B_scales = w1s_scales;
    a.out = w.Hb;
    ce = launch_grouped_gemm(a, sms, s);
    if (ce == cudaSuccess)
      ce = launch_quant_row(static_cast<const uint16_t *>(w.Hb), nullptr, M, Ns,
                            static_cast<uint8_t *>(w.H), w.Hs, sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
    a.mode = kDown;
    a.A = w.H;
    a.A_scales = w.Hs;
    a.B = w2s;
    a.B_scales = w2s_scales;
    a.out = out_shared;
    return from_cuda(launch_grouped_gemm(a, sms, s));
  }
  if (fp8) {
    // x in 1 x 128 groups, its scales moved to the GEMM's group-major layout
    ce = launch_quant_group(x, nullptr, M, K, static_cast<uint8_t *>(w.xq), w.xs_rows, sms, s);
    if (ce == cudaSuccess)
      ce = launch_scales_group_major(w.xs_rows, M, K / 128, w.xs, scale_ld((size_t)M), sms, s);
    if (ce != cudaSuccess) return from_cuda(ce);
    a.A = w.xq;
    a.A_scales = w.xs;
    a.scale_ld = scale_ld((size_t)M);
    a.B_scales = w1s_scales;
    a.out_scales = w.Hs;
  }
  ce = launch_grouped_gemm(a, sms, s);
  if (ce != cudaSuccess) return from_cuda(ce);
  a.mode = kDown;
  a.A = w.H;
  a.A_scales = w.Hs;
  a.B = w2s;
  a.B_scales = w2s_scales;
  a.out_scales = nullptr;
  a.out = out_shared;
  return from_cuda(launch_grouped_gemm(a, sms, s));
}

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
                                  struct CUevent_st *ev_input_ready,
                                  struct CUevent_st *ev_output_ready) {
  // every argument is checked before anything is enqueued
  gbmoe_status_t st = forward_validate(x, logits, bias, M, K, N, E_global, expert_map, E,
                                       topk, score_fn, n_groups, topk_groups,
                                       apply_router_weight_on_input, activation, dtype, w1,
                                       w1_scales, w2, w2_scales, a1_scale, a2_scale, out, ws,
                                       ws_bytes);
  if (st != GBMOE_OK) return st;
  st = shared_validate(x, M, K, Ns, w1s, w1s_scales, w2s, w2s_scales, shared_dtype, activation,
                       out_shared, ws_shared, ws_shared_bytes);
  if (st != GBMOE_OK) return st;
  if (aux_stream && (!ev_input_ready || !ev_output_ready)) return GBMOE_INVALID_ARG;
  int sms;
  st = device_info(&sms);
  if (st != GBMOE_OK || M == 0) return st;
  cudaStream_t s = (cudaStream_t)stream;
  cudaStream_t aux = (cudaStream_t)aux_stream;
  cudaEvent_t ev_in = (cudaEvent_t)ev_input_ready, ev_out = (cudaEvent_t)ev_output_ready;
  if (aux) {
    // fork: the shared experts on aux_stream once `stream` reaches this point
    cudaError_t ce = cudaEventRecord(ev_in, s);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(aux, ev_in, 0);
    if (ce != cudaSuccess) return from_cuda(ce);
    gbmoe_status_t st1 = moe_shared_expert_forward(x, M, K, Ns, w1s, w1s_scales, w2s,
                                                   w2s_scales, shared_dtype, activation,
                                                   out_shared, ws_shared, ws_shared_bytes,
                                                   err_word, aux_stream);
    cudaError_t ce1 = cudaEventRecord(ev_out, aux);
    // the routed experts on `stream` meanwhile
    gbmoe_status_t st2 = moe_forward(x, logits, bias, M, K, N, E_global, expert_map, E, topk,
                                     score_fn, n_groups, topk_groups, renormalize,
                                     apply_router_weight_on_input, activation, dtype, w1,
                                     w1_scales, w2, w2_scales, a1_scale, a2_scale, out, nullptr,
                                     nullptr, ws, ws_bytes, err_word, stream);
    // join (always, so that `stream` never runs ahead of aux_stream's work)
    cudaError_t ce2 = ce1 == cudaSuccess ? cudaStreamWaitEvent(s, ev_out, 0) : ce1;
    if (st1 != GBMOE_OK) return st1;
    if (st2 != GBMOE_OK) return st2;
    return from_cuda(ce2);
  }
  st = moe_shared_expert_forward(x, M, K, Ns, w1s, w1s_scales, w2s, w2s_scales, shared_dtype,
                                 activation, out_shared, ws_shared, ws_shared_bytes, err_word,
                                 stream);
  if (st != GBMOE_OK) return st;
  return moe_forward(x, logits, bias, M, K, N, E_global, expert_map, E, topk, score_fn,
                     n_groups, topk_groups, renormalize, apply_router_weight_on_input,
                     activation, dtype, w1, w1_scales, w2, w2_scales, a1_scale, a2_scale, out,
                     nullptr, nullptr, ws, ws_bytes, err_word, stream);
}

}  // extern "C"

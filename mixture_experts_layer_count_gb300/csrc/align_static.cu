// align_static.cu -- moe_align_permute_no_ws: the stable counting sort of
// moe_align_permute for callers that cannot hand the library any scratch
// memory.  Its per-chunk histograms live in a fixed array in device global
// memory that belongs to this library (loaded with it, held by every GPU
// that loads the library until the process exits) instead of a caller
// workspace.  The kernels are the ones moe_align_permute launches.
#include <cstdint>
#include <mutex>

#include "gbmoe.h"
#include "kernels.h"

namespace gbmoe {
namespace {

// int32 entries: 65536 x 4 B = 256 KiB.  The sort needs one histogram of E
// entries per chunk of 2048 pairs, so chunks * E must stay within this.
constexpr int kNoWsHistEntries = 65536;
constexpr int kMaxExpertsNoWs = 512;
constexpr int kMaxDevicesNoWs = 64;

__device__ __align__(256) int32_t g_align_hist[kNoWsHistEntries];

// Device address of g_align_hist, looked up once per device.  In host code
// the symbol name is only a host-side stand-in for the array, not a device
// address, so the kernels are given the address cudaGetSymbolAddress returns.
int32_t *g_hist_addr[kMaxDevicesNoWs] = {};
std::mutex g_hist_mu;

gbmoe_status_t hist_address(int32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNoWs)
    return GBMOE_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_hist_mu);
  if (g_hist_addr[dev] == nullptr) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return GBMOE_UNSUPPORTED;
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_align_hist);
    if (e != cudaSuccess || p == nullptr) return status_from_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_hist_addr[dev] = static_cast<int32_t *>(p);
  }
  *out = g_hist_addr[dev];
  return GBMOE_OK;
}

}  // namespace
}  // namespace gbmoe

extern "C" gbmoe_status_t moe_align_permute_no_ws(const int32_t *topk_ids, int M,
                                                  int topk, int E, int32_t *counts,
                                                  int32_t *offsets,
                                                  int32_t *sorted_pair_ids,
                                                  int32_t *inv, int32_t *err_word,
                                                  gbmoe_stream_t stream) {
  using namespace gbmoe;
  if (M < 0 || topk < 1 || E < 1 || E > kMaxExpertsNoWs || !offsets) return GBMOE_INVALID_ARG;
  if ((size_t)M * topk > (size_t)INT32_MAX) return GBMOE_INVALID_ARG;
  if (M > 0 && (!topk_ids || !sorted_pair_ids || !inv)) return GBMOE_INVALID_ARG;
  const int P = M * topk;
  if ((long long)align_num_chunks(P) * E > kNoWsHistEntries) return GBMOE_INVALID_ARG;
  int32_t *hist = nullptr;
  gbmoe_status_t st = hist_address(&hist);
  if (st != GBMOE_OK) return st;
  // the address above is the current device's copy of the array: a stream
  // of another device would have its kernels write through it
  if (stream != nullptr) {
    int cur = -1, sdev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess ||
        cudaStreamGetDevice((cudaStream_t)stream, &sdev) != cudaSuccess || sdev != cur)
      return GBMOE_INVALID_ARG;
  }
  return status_from_cuda(launch_align(topk_ids, P, E, nullptr, E, counts, offsets,
                                       sorted_pair_ids, inv, hist, err_word,
                                       (cudaStream_t)stream));
}

// gemm2sm.cu -- the bf16 grouped GEMMs on CTA pairs: tcgen05.mma with
// cta_group::2 computes a 256 x 256 tile on two SMs (M = 256 rows of A split
// 128 / 128 between the pair, the 256 rows of the B tile split the same way,
// each SM's TMEM receiving its 128 rows of the fp32 accumulator).
//
// The same computation as gemm.cu (gate/up + SiLU*mul or GELU*mul, down +
// router weight; Standard, BatchedExperts and dense row groups), organised so
// that each SM stages half of the B tile: per K block of 64 an SM moves
// 16 KB of A and 16 KB of B through shared memory instead of 16 + 32 KB,
// which leaves the shared-memory bandwidth to the tensor core.
//
// Roles in each CTA of the pair (192 threads):
//   warp 0 (one lane)  TMA producer of this CTA's halves; all copies of a
//                      stage complete the transaction of the even CTA's
//                      full barrier
//   warp 1             TMEM allocation (both CTAs, cta_group::2); in the even
//                      CTA one lane issues the MMAs and commits them to the
//                      barriers of both CTAs (multicast)
//   warps 2..5         epilogue on this CTA's 128 rows; TMEM-free signals go
//                      to the even CTA's barrier
// Every mbarrier wait is bounded (2 s); on expiry the kernel records
// GBMOE_ERR_TIMEOUT and leaves its loops.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "per_device.h"

namespace gbmoe {

namespace {

using namespace gemm;

constexpr int kPairBM = 256;                // rows per pair tile
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kBK = kBKB / 2;               // bf16 elements per stage row
constexpr int kMmaPerStage = kBK / 16;
constexpr int kStages2 = 6;
constexpr int kAHalf = 128 * kBKB;          // 16 KB: this CTA's 128 rows of A
constexpr int kBHalf = 128 * kBKB;          // 16 KB: this CTA's 128 rows of B
constexpr uint32_t kIdesc = umma_idesc(kPairBM, kBN, kFmtBF16);

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages2 * kAHalf;
constexpr int kOffBar = kOffB + kStages2 * kBHalf;   // 196608
constexpr int kNumBars = 2 * kStages2 + 2 + 2 + 1;   // full, empty, tfull, tempty, done
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kOffPrefix = kOffTmem + 16;
constexpr int kOffRBase = kOffPrefix + (kMaxE + 1) * 4;
constexpr int kOffRCnt = kOffRBase + kMaxE * 4;
constexpr int kSmemUsed = kOffRCnt + kMaxE * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;

struct KParams {
  const int32_t *offsets;
  const int32_t *counts;
  int E, T, N, K;
  int n_tiles;
  int num_kb;
  int b_rows;
  void *out;
  const int32_t *sorted;
  const float *topk_w;
  int32_t *err;
};

template <int MODE, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw_u32);

  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const bool leader = rank == 0;
  const uint32_t sA = base + kOffA;
  const uint32_t sB = base + kOffB;
  const uint32_t bar0 = base + kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages2 + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages2 + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages2 + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kStages2 + 4);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + kOffTmem);
  int *prefix = reinterpret_cast<int *>(sbase + kOffPrefix);
  int *rbase = reinterpret_cast<int *>(sbase + kOffRBase);
  int *rcnt = reinterpret_cast<int *>(sbase + kOffRCnt);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  tile_table_fill(p.offsets, p.counts, E, p.T, p.n_tiles, prefix, rbase, rcnt, p.err, kPairBM);
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(full_bar(s), 1);    // the even CTA's producer (expect_tx for both CTAs)
      mbar_init(empty_bar(s), 1);   // the pair's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * kEpiWarps);  // epilogue warps of both CTAs
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc_pair<512>(smem_u32(tmem_slot));
  __syncthreads();
  if (warp == 0) tile_table_scan(prefix, E, lane);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = prefix[E];
  const int num_kb = p.num_kb;

  if (warp == 0) {
    // =========================== TMA producer ===========================
    if (lane == 0) {
      int it = 0;
      int last_round[kStages2];
#pragma unroll
      for (int s = 0; s < kStages2; ++s) last_round[s] = -1;
      bool ok = true;
      for (int tile = pair_id; tile < total && ok; tile += n_pairs) {
        int e, mt, nt;
        decode_tile(prefix, E, p.n_tiles, tile, e, mt, nt);
        const int a_row = rbase[e] + mt * kPairBM + 128 * (int)rank;
        int b_row;
        if (MODE == kGateUpMode)  // the even CTA stages the gate rows, the odd one the up rows
          b_row = e * p.b_rows + (rank ? p.N : 0) + nt * 128;
        else
          b_row = e * p.b_rows + nt * kBN + 128 * (int)rank;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages2, round = it / kStages2;
          if (!mbar_wait(empty_bar(s), (round & 1) ^ 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(full_bar(s), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * (kAHalf + kBHalf));
          const int x = kb * kBK;
          tma_load_2d_pair(sA + s * kAHalf, &tmA, fb, x, a_row);
          tma_load_2d_pair(sB + s * kBHalf, &tmB, fb, x, b_row);
          last_round[s] = round;
        }
      }
      // Copies still in flight land before the CTA can leave.  The odd CTA's
      // copies complete the even CTA's full barrier, which it cannot wait
      // on, so both CTAs wait (bounded) until the pair's MMA has released
      // each stage they loaded last: the MMA issuer waited for those bytes
      // first.  The even CTA also waits for its full barriers, which count
      // the bytes of both CTAs; it stays resident (final cluster barrier)
      // until it has.  After a timeout these waits end within their own
      // limit, by which time copies issued before the stall have landed.
#pragma unroll
      for (int s = 0; s < kStages2; ++s) {
        if (last_round[s] < 0) continue;
        if (leader) mbar_wait(full_bar(s), last_round[s] & 1, 100000000ull);
        mbar_wait(empty_bar(s), last_round[s] & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // =========================== MMA issuer =============================
    if (leader && lane == 0) {
      int it = 0, acc_it = 0;
      bool ok = true;
      for (int tile = pair_id; tile < total && ok; tile += n_pairs) {
        const int buf = acc_it & 1, use = acc_it >> 1;
        if (!mbar_wait_cluster(tempty_bar(buf), (use & 1) ^ 1)) {
          set_err(p.err, GBMOE_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBN;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages2, round = it / kStages2;
          if (!mbar_wait_cluster(full_bar(s), round & 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = umma_desc_sw128(sA + s * kAHalf);
          const uint64_t db = umma_desc_sw128(sB + s * kBHalf);
#pragma unroll
          for (int k = 0; k < kMmaPerStage; ++k)
            umma_f16_pair(d, da + 2 * k, db + 2 * k, kIdesc, (kb | k) != 0);
          umma_commit_pair_mc(empty_bar(s), 0x3);
        }
        if (!ok) break;
        umma_commit_pair_mc(tfull_bar(buf), 0x3);
        ++acc_it;
      }
      umma_commit_pair(done_bar);
      mbar_wait(done_bar, 0, 100000000ull);
    }
  } else {
    // ============================= epilogue =============================
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    const uint32_t t_lane = (uint32_t)(q * 32) << 16;
    int acc_it = 0;
    for (int tile = pair_id; tile < total; tile += n_pairs) {
      int e, mt, nt;
      decode_tile(prefix, E, p.n_tiles, tile, e, mt, nt);
      const int r = mt * kPairBM + 128 * (int)rank + row_in_tile;  // row within the expert
      const bool valid = r < rcnt[e];
      const int arow = rbase[e] + r;
      const int buf = acc_it & 1, use = acc_it >> 1;
      if (!mbar_wait(tfull_bar(buf), use & 1)) {
        set_err(p.err, GBMOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + t_lane + buf * kBN;
      if (MODE == kGateUpMode) {
        uint16_t *hrow = static_cast<uint16_t *>(p.out) + (size_t)arow * p.N + nt * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c * 32, g);
          tmem_ld32(tb + 128 + c * 32, u);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = gate_act<ACT>(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
            const float h1 =
                gate_act<ACT>(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
            pk[i] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(hrow + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        size_t orow = 0;
        float w = 1.0f;
        if (valid) {
          if (p.sorted) {
            const int pair = p.sorted[arow];
            orow = (size_t)pair;
            w = p.topk_w ? p.topk_w[pair] : 1.0f;
          } else {
            orow = (size_t)arow;
          }
        }
        uint16_t *yrow = static_cast<uint16_t *>(p.out) + orow * p.K + nt * kBN;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          if (nt * kBN + c * 32 >= p.K) break;  // uniform across the warp
          uint32_t v[32];
          tmem_ld32(tb + c * 32, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(w * __uint_as_float(v[2 * i]), w * __uint_as_float(v[2 * i + 1]));
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(yrow + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(buf), 0));
      ++acc_it;
    }
  }

  // all MMAs are done (the epilogues consumed every tile) before TMEM goes
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair<512>(tmem_base);
}

template <int MODE, int ACT>
cudaError_t launch_pair(const GroupedGemmArgs &a, int num_sms, cudaStream_t s) {
  static PerDeviceInt smem_set;
  cudaError_t st = set_smem_once(smem_set, grouped_gemm_pair_kernel<MODE, ACT>, kSmemBytes);
  if (st != cudaSuccess) return st;
  const bool gate_up = MODE == kGateUpMode;
  const int Kd = gate_up ? a.K : a.N;
  const int b_rows = gate_up ? 2 * a.N : a.K;
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, a.A, kTmapBF16, (uint64_t)Kd, (uint64_t)a.a_rows,
                      (uint64_t)Kd * 2, kBK, 128, true) ||
      !encode_tmap_2d(&tmB, a.B, kTmapBF16, (uint64_t)Kd, (uint64_t)a.E * b_rows,
                      (uint64_t)Kd * 2, kBK, 128, true))
    return cudaErrorInvalidValue;
  KParams p;
  p.offsets = a.offsets;
  p.counts = a.counts;
  p.E = a.E;
  p.T = a.T;
  p.N = a.N;
  p.K = a.K;
  p.n_tiles = gate_up ? a.N / 128 : (a.K + kBN - 1) / kBN;
  p.num_kb = Kd / kBK;
  p.b_rows = b_rows;
  p.out = a.out;
  p.sorted = a.sorted_pair_ids;
  p.topk_w = a.topk_weights;
  p.err = a.err;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent: as many pairs as can be resident at once (an SM left without
  // a partner in its GPC hosts none)
  static PerDeviceInt resident;
  int resident_pairs = 0;
  st = resident.get(&resident_pairs, [&](int *v) {
    cfg.gridDim = dim3(2 * (num_sms / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<MODE, ACT>, &cfg) !=
            cudaSuccess ||
        n < 1) {
      cudaGetLastError();  // the query's error, if any, is not a launch error
      n = num_sms / 2;
    }
    *v = n;
    return cudaSuccess;
  });
  if (st != cudaSuccess) return st;
  const long long mtiles = a.offsets ? (a.a_rows + kPairBM - 1) / kPairBM + a.E
                                     : (long long)a.E * ((a.T + kPairBM - 1) / kPairBM);
  const long long tiles = mtiles * p.n_tiles;
  const int pairs = (int)(tiles < resident_pairs ? tiles : resident_pairs);
  cfg.gridDim = dim3(2 * (pairs < 1 ? 1 : pairs));
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE, ACT>, tmA, tmB, p);
}

}  // namespace

cudaError_t launch_grouped_gemm_pair(const GroupedGemmArgs &a, int num_sms, cudaStream_t s) {
  if (a.mode == kDown) return launch_pair<kDownMode, kActSilu>(a, num_sms, s);
  return a.act == GBMOE_ACT_GELU ? launch_pair<kGateUpMode, kActGelu>(a, num_sms, s)
                                 : launch_pair<kGateUpMode, kActSilu>(a, num_sms, s);
}

}  // namespace gbmoe

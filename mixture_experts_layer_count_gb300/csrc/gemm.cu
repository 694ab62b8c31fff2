// gemm.cu -- the two expert GEMMs of [Permute-Experts-Unpermute] in bf16, or
// in e4m3 with one scale per row of each operand (per-token activations,
// per-channel weights), as grouped GEMMs on the sm_103a tensor cores
// (tcgen05.mma, fp32 accumulators in TMEM), operands staged in shared memory
// by TMA; plus the tensor-map encoder and the dispatch between the kernels.
// With per-row scales the whole K accumulates in TMEM and the epilogue
// applies s_a[row] * s_w[column] once (the 1 x 128 / 128 x 128 block-scaled
// e4m3 GEMMs are in gemm_fp8.cu).
//
// In "vllm/model_executor/layers/fused_moe/modular_kernel.py"
// (FusedMoEPermuteExpertsUnpermute, its apply), the experts stage is two
// GEMMs with the gated activation and an optional requantisation between
// them: the gate/up GEMM with w1 (E, 2N, K) feeds the gated activation
// (silu_and_mul, output half as wide), the down
// GEMM with w2 (E, K, N) gives the per-pair expert output that [Finalize]
// weights and reduces.  Here:
//   gate/up: H[i, n] = silu(A[i] . w1[e, n]) * (A[i] . w1[e, N + n])
//   down:    y[row(i), k] = weight(i) * (H[i] . w2[e, k])
// for the rows i of each expert e.  Rows of an expert are contiguous in A:
// Standard format [offsets[e], offsets[e+1]); BatchedExperts format
// [e*T, e*T + min(counts[e], T)), the device-resident counts of "EP:
// CUDA-graph-safe HT internode dispatch+combine (worst-tokens mode)", read on
// the device only.
//
// Kernel shape (one persistent CTA per SM, warp-specialised, 192 threads):
//   warp 0 (one lane)  TMA producer: A tile 128 x 128 B, B tile 256 x 128 B per
//                      stage, 4 stages, 128-byte swizzle
//   warp 1             TMEM allocation; one lane issues tcgen05.mma
//                      (M 128, N 256, K 16, fp32 accumulators in TMEM)
//   warps 2..5         epilogue: tcgen05.ld, SiLU*mul or weighting, stores
// Two 256-column TMEM accumulators let the epilogue of one tile overlap the
// mainloop of the next.  Every wait is bounded (2 s); on expiry the kernel
// sets GBMOE_ERR_TIMEOUT, leaves its loops, waits (bounded) for its copies
// and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "gemm_common.cuh"
#include "kernels.h"
#include "per_device.h"

namespace gbmoe {

namespace {

using namespace gemm;

constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
// a stage row is kBKB = 128 bytes of K: 64 bf16 or 128 e4m3 elements, four
// MMAs either way (kind::f16 has K = 16, kind::f8f6f4 K = 32)
template <bool F8>
__host__ __device__ constexpr int stage_k() { return F8 ? kBKB : kBKB / 2; }
constexpr int kMmaPerStage = 4;
template <bool F8>
__host__ __device__ constexpr uint32_t idesc_of() { return umma_idesc(kBM, kBN, F8 ? kFmtE4M3 : kFmtBF16); }

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kAStage;
constexpr int kOffBar = kOffB + kStages * kBStage;     // 196608
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;      // full, empty, tfull, tempty, done
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kOffPrefix = kOffTmem + 16;
constexpr int kOffRBase = kOffPrefix + (kMaxE + 1) * 4;
constexpr int kOffRCnt = kOffRBase + kMaxE * 4;
constexpr int kSmemUsed = kOffRCnt + kMaxE * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;           // slack for the 1024 alignment

struct KParams {
  const int32_t *offsets;   // Standard
  const int32_t *counts;    // Batched
  int E, T, N, K;
  int n_tiles;              // output tiles per expert along the GEMM's N
  int num_kb;               // K blocks (of kBKB bytes)
  int b_rows;               // rows of B per expert (2N or K)
  void *out;
  const int32_t *sorted;    // down, Standard
  const float *topk_w;      // down, Standard
  const float *a_scales;    // e4m3: one per row of A
  const float *b_scales;    // e4m3: one per row of B (E * b_rows)
  int32_t *err;
};

// the 32 per-row weight scales of output columns [col, col + 32) of expert e
// (every lane reads the same addresses: broadcast loads)
__device__ __forceinline__ void load_scales32(const float *b_scales, size_t first, float (&w)[32]) {
  const float4 *p4 = reinterpret_cast<const float4 *>(b_scales + first);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = __ldg(p4 + i);
    w[4 * i] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
}

template <int MODE, int ACT, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw_u32);

  const uint32_t sA = base + kOffA;
  const uint32_t sB = base + kOffB;
  const uint32_t bar0 = base + kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kStages + 4);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + kOffTmem);
  int *prefix = reinterpret_cast<int *>(sbase + kOffPrefix);
  int *rbase = reinterpret_cast<int *>(sbase + kOffRBase);
  int *rcnt = reinterpret_cast<int *>(sbase + kOffRCnt);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  tile_table_fill(p.offsets, p.counts, E, p.T, p.n_tiles, prefix, rbase, rcnt, p.err);
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc<512>(smem_u32(tmem_slot));
  __syncthreads();
  if (warp == 0) tile_table_scan(prefix, E, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = prefix[E];
  const int num_kb = p.num_kb;

  if (warp == 0) {
    // =========================== TMA producer ===========================
    if (lane == 0) {
      int it = 0;
      int last_round[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_round[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int e, mt, nt;
        decode_tile(prefix, E, p.n_tiles, tile, e, mt, nt);
        const int a_row = rbase[e] + mt * kBM;
        int b_row0, b_row1;
        if (MODE == kGateUpMode) {
          b_row0 = e * p.b_rows + nt * 128;
          b_row1 = e * p.b_rows + p.N + nt * 128;
        } else {
          b_row0 = e * p.b_rows + nt * kBN;
          b_row1 = b_row0 + 128;
        }
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages, round = it / kStages;
          if (!mbar_wait(empty_bar(s), (round & 1) ^ 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), kAStage + kBStage);
          const int x = kb * stage_k<F8>();
          tma_load_2d(sA + s * kAStage, &tmA, full_bar(s), x, a_row);
          tma_load_2d(sB + s * kBStage, &tmB, full_bar(s), x, b_row0);
          tma_load_2d(sB + s * kBStage + kBStage / 2, &tmB, full_bar(s), x, b_row1);
          last_round[s] = round;
        }
      }
      // copies still in flight land before the CTA can leave
#pragma unroll
      for (int s = 0; s < kStages; ++s)
        if (last_round[s] >= 0) mbar_wait(full_bar(s), last_round[s] & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer =============================
    if (lane == 0) {
      int it = 0, acc_it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const int buf = acc_it & 1, use = acc_it >> 1;
        if (!mbar_wait(tempty_bar(buf), (use & 1) ^ 1)) {
          set_err(p.err, GBMOE_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBN;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages, round = it / kStages;
          if (!mbar_wait(full_bar(s), round & 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = umma_desc_sw128(sA + s * kAStage);
          const uint64_t db = umma_desc_sw128(sB + s * kBStage);
#pragma unroll
          for (int k = 0; k < kMmaPerStage; ++k) {
            if (F8)
              umma_f8(d, da + 2 * k, db + 2 * k, idesc_of<F8>(), (kb | k) != 0);
            else
              umma_f16(d, da + 2 * k, db + 2 * k, idesc_of<F8>(), (kb | k) != 0);
          }
          umma_commit(empty_bar(s));
        }
        if (!ok) break;
        umma_commit(tfull_bar(buf));
        ++acc_it;
      }
      // every MMA issued above has finished before TMEM is released
      umma_commit(done_bar);
      mbar_wait(done_bar, 0, 100000000ull);
    }
  } else {
    // ============================= epilogue =============================
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row_in_tile = q * 32 + lane;
    const uint32_t t_lane = (uint32_t)(q * 32) << 16;
    int acc_it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, mt, nt;
      decode_tile(prefix, E, p.n_tiles, tile, e, mt, nt);
      const int r = mt * kBM + row_in_tile;  // row within the expert
      const bool valid = r < rcnt[e];
      const int arow = rbase[e] + r;         // row of A / H
      const int buf = acc_it & 1, use = acc_it >> 1;
      if (!mbar_wait(tfull_bar(buf), use & 1)) {
        set_err(p.err, GBMOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + t_lane + buf * kBN;
      const float sa = F8 && valid ? p.a_scales[arow] : 1.0f;
      if (MODE == kGateUpMode) {
        uint16_t *hrow = static_cast<uint16_t *>(p.out) + (size_t)arow * p.N + nt * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c * 32, g);
          tmem_ld32(tb + 128 + c * 32, u);
          tmem_ld_wait();
          if (F8) {  // g, u *= s_a[row] * s_w[column]
            float sw[32];
            const size_t col = (size_t)e * p.b_rows + nt * 128 + c * 32;
            load_scales32(p.b_scales, col, sw);
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = __float_as_uint(__uint_as_float(g[i]) * (sa * sw[i]));
            load_scales32(p.b_scales, col + p.N, sw);
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * (sa * sw[i]));
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = gate_act<ACT>(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
            const float h1 = gate_act<ACT>(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
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
          if (F8) {  // y *= s_a[row] * s_w[column]
            float sw[32];
            load_scales32(p.b_scales, (size_t)e * p.b_rows + nt * kBN + c * 32, sw);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * (sa * sw[i]));
          }
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
      if (lane == 0) mbar_arrive(tempty_bar(buf));
      ++acc_it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<512>(tmem_base);
}

// cuTensorMapEncodeTiled, resolved through the runtime (no -lcuda link)
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

// looked up once per process (the CUDA driver API entry point is not per
// device);
// std::call_once makes concurrent first calls from several threads safe
bool resolve_encode() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode != nullptr;
}

template <int MODE, int ACT, bool F8>
cudaError_t launch_bf16(const GroupedGemmArgs &a, int num_sms, cudaStream_t s) {
  static PerDeviceInt smem_set;
  cudaError_t st = set_smem_once(smem_set, grouped_gemm_kernel<MODE, ACT, F8>, kSmemBytes);
  if (st != cudaSuccess) return st;
  const bool gate_up = MODE == kGateUpMode;
  const int Kd = gate_up ? a.K : a.N;          // contraction length
  const int b_rows = gate_up ? 2 * a.N : a.K;  // rows of B per expert
  const int esz = F8 ? 1 : 2;                  // bytes per element
  const int kind = F8 ? kTmapU8 : kTmapBF16;
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, a.A, kind, (uint64_t)Kd, (uint64_t)a.a_rows,
                      (uint64_t)Kd * esz, stage_k<F8>(), kBM, true) ||
      !encode_tmap_2d(&tmB, a.B, kind, (uint64_t)Kd, (uint64_t)a.E * b_rows,
                      (uint64_t)Kd * esz, stage_k<F8>(), 128, true))
    return cudaErrorInvalidValue;
  KParams p;
  p.offsets = a.offsets;
  p.counts = a.counts;
  p.E = a.E;
  p.T = a.T;
  p.N = a.N;
  p.K = a.K;
  p.n_tiles = gate_up ? a.N / 128 : (a.K + kBN - 1) / kBN;
  p.num_kb = Kd / stage_k<F8>();
  p.b_rows = b_rows;
  p.out = a.out;
  p.sorted = a.sorted_pair_ids;
  p.topk_w = a.topk_weights;
  p.a_scales = a.A_scales;
  p.b_scales = a.B_scales;
  p.err = a.err;
  // upper bound on the tiles: every expert may end with a partial m-tile
  long long mtiles = a.offsets ? (a.a_rows + kBM - 1) / kBM + a.E
                               : (long long)a.E * ((a.T + kBM - 1) / kBM);  // batched / dense
  long long tiles = mtiles * p.n_tiles;
  int grid = (int)(tiles < num_sms ? tiles : num_sms);
  if (grid < 1) grid = 1;
  grouped_gemm_kernel<MODE, ACT, F8><<<grid, kThreads, kSmemBytes, s>>>(tmA, tmB, p);
  return cudaGetLastError();
}

}  // namespace

bool encode_tmap_2d(CUtensorMap *map, const void *base, int kind, uint64_t cols,
                    uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols,
                    uint32_t box_rows, bool swizzle128) {
  if (!resolve_encode()) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (kind == kTmapBF16) dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  else if (kind == kTmapF32) dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool bf16_uses_cta_pairs(const GroupedGemmArgs &a) {
  // Row capacity the launch covers: Standard format the M*topk permuted rows,
  // BatchedExperts / dense E*T.  CTA pairs (256-row tiles) when the experts
  // average 128 rows or more; below that a pair tile is mostly padding, and
  // the 1-SM kernel keeps more weight bytes in flight per SM (4 stages x
  // 32 KB of B against 6 x 16 KB), which is what a weight-streaming launch
  // (decode) needs.  e4m3 operands stay on one SM: a 128-byte K block is
  // twice the MMA work of a bf16 one, so the 1-SM stage traffic (48 KB per
  // 512 MMA cycles) is already below what shared memory delivers, and the
  // weight tiles mostly stream from HBM.
  if (a.fp8ch) return false;
  const long long rows = a.offsets ? (long long)a.a_rows : (long long)a.T * a.E;
  return rows >= 128LL * a.E;
}

template <bool F8>
cudaError_t launch_one_sm(const GroupedGemmArgs &a, int num_sms, cudaStream_t s) {
  if (a.mode == kDown) return launch_bf16<kDownMode, kActSilu, F8>(a, num_sms, s);
  return a.act == GBMOE_ACT_GELU ? launch_bf16<kGateUpMode, kActGelu, F8>(a, num_sms, s)
                                 : launch_bf16<kGateUpMode, kActSilu, F8>(a, num_sms, s);
}

cudaError_t launch_grouped_gemm(const GroupedGemmArgs &a, int num_sms,
                                cudaStream_t s) {
  if (a.fp8) return launch_grouped_gemm_fp8(a, num_sms, s);
  if (bf16_uses_cta_pairs(a)) return launch_grouped_gemm_pair(a, num_sms, s);
  return a.fp8ch ? launch_one_sm<true>(a, num_sms, s) : launch_one_sm<false>(a, num_sms, s);
}

}  // namespace gbmoe

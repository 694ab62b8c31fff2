// gemm.cu -- the two expert GEMMs of [Permute-Experts-Unpermute] as grouped
// GEMMs on the sm_103a tensor cores (tcgen05.mma, accumulators in TMEM),
// operands staged in shared memory by TMA.
//
// FusedMoEPermuteExpertsUnpermute.apply in
// "vllm/model_executor/layers/fused_moe/modular_kernel.py" is "matmul +
// act_mul + optionally quant + matmul": the gate/up GEMM with w1 (E, 2N, K)
// feeds the gated activation (silu_and_mul, output half as wide), the down
// GEMM with w2 (E, K, N) gives the per-pair expert output that [Finalize]
// weights and reduces.  Here:
//   kGateUp: H[i, n] = silu(A[i] . w1[e, n]) * (A[i] . w1[e, N + n])   (+ e4m3 requant)
//   kDown:   y[row(i), k] = weight(i) * (H[i] . w2[e, k])
// for the rows i of each expert e.  Rows of an expert are contiguous in A:
// Standard format [offsets[e], offsets[e+1]); BatchedExperts format
// [e*T, e*T + min(counts[e], T)), the device-resident counts of "EP:
// CUDA-graph-safe HT internode dispatch+combine (worst-tokens mode)", read on
// the device only.
//
// Kernel shape (one persistent CTA per SM, warp-specialised):
//   warp 0 (one lane)  TMA producer: A tile 128 x 128 B, B tile 256 x 128 B per
//                      stage, 4 stages, 128-byte swizzle
//   warp 1             TMEM allocation; one lane issues tcgen05.mma
//                      (M 128, N 256, fp32 accumulators in TMEM)
//   warps 2..          epilogue: tcgen05.ld, SiLU*mul or weighting, stores
// bf16: two 256-column TMEM accumulators, so the epilogue of one tile overlaps
//   the mainloop of the next.
// fp8: the per-128-K block scales (1 x 128 activations, 128 x 128 weights, fp32)
//   change along K, so each K block is accumulated alone in TMEM (two
//   buffers) and the epilogue warps promote it into fp32 registers:
//   acc += s_a[row, kb] * s_w[blk, kb] * partial.
// Tiles are ordered (expert, n-tile, m-tile) with m fastest, so CTAs that run
// at the same time share weight tiles through L2.
// Every wait is bounded (2 s); on expiry the kernel sets GBMOE_ERR_TIMEOUT,
// leaves its loops, waits (bounded) for its copies and MMAs in flight, frees
// TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbmoe {

namespace {

constexpr int kBM = 128;     // rows per tile (UMMA M)
constexpr int kBN = 256;     // output columns per tile (UMMA N)
constexpr int kBKB = 128;    // K bytes per stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBKB;  // 16 KB
constexpr int kBStage = kBN * kBKB;  // 32 KB
constexpr int kMaxE = 512;

template <bool FP8>
struct Cfg {
  static constexpr int kEpiWarps = FP8 ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kKPerMma = FP8 ? 32 : 16;          // K elements per tcgen05.mma
  static constexpr int kElemBytes = FP8 ? 1 : 2;
  static constexpr int kBK = kBKB / kElemBytes;           // K elements per stage
  static constexpr int kMmaPerStage = kBK / kKPerMma;     // 4
  static constexpr uint32_t kIdesc =
      umma_idesc(kBM, kBN, FP8 ? kFmtE4M3 : kFmtBF16);
};

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kAStage;
constexpr int kOffBar = kOffB + kStages * kBStage;       // 196608
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 2;    // full, empty, tfull, tempty, done, xchg
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kOffAmax = kOffTmem + 16;                  // fp8 requant exchange [2][2][128] f32
constexpr int kOffPrefix = kOffAmax + 2 * 2 * 128 * 4;
constexpr int kOffRBase = kOffPrefix + (kMaxE + 1) * 4;
constexpr int kOffRCnt = kOffRBase + kMaxE * 4;
constexpr int kSmemUsed = kOffRCnt + kMaxE * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;             // slack for the 1024 alignment

struct KParams {
  int mode;
  const int32_t *offsets;   // Standard
  const int32_t *counts;    // Batched
  int E, T, N, K;
  int n_tiles;              // output tiles per expert along the GEMM's N
  int num_kb;               // K blocks (of kBKB bytes)
  int a_rows;               // rows of A's allocation
  int b_rows;               // rows of B per expert (2N or K)
  void *out;
  float *out_scales;        // fp8 gate-up: (a_rows, N/128)
  const float *a_scales;    // fp8: (a_rows, num_kb)
  const float *b_scales;    // fp8: (E, b_rows/128, num_kb)
  const int32_t *sorted;    // down, Standard
  const float *topk_w;      // down, Standard
  int32_t *err;
};

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

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3) |
         ((uint32_t)__nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3) << 8) |
         ((uint32_t)__nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3) << 16) |
         ((uint32_t)__nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3) << 24);
}

template <bool FP8>
__global__ void __launch_bounds__(Cfg<FP8>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const KParams p) {
  using C = Cfg<FP8>;
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
  auto xchg_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 5 + b); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + kOffTmem);
  float *amax_x = reinterpret_cast<float *>(sbase + kOffAmax);  // [2 bufs][2 halves][128]
  int *prefix = reinterpret_cast<int *>(sbase + kOffPrefix);
  int *rbase = reinterpret_cast<int *>(sbase + kOffRBase);
  int *rcnt = reinterpret_cast<int *>(sbase + kOffRCnt);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int E = p.E;

  // ---- prologue: rows of each expert and the tile prefix sums
  for (int e = tid; e < E; e += blockDim.x) {
    int b, r;
    if (p.offsets) {
      b = p.offsets[e];
      r = p.offsets[e + 1] - b;
    } else {
      r = p.counts[e];
      if (r < 0 || r > p.T) {
        if (blockIdx.x == 0) set_err(p.err, GBMOE_ERR_COUNT_RANGE);
        r = r < 0 ? 0 : p.T;
      }
      b = e * p.T;
    }
    rbase[e] = b;
    rcnt[e] = r;
    prefix[e + 1] = ((r + kBM - 1) / kBM) * p.n_tiles;
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::kEpiWarps);
      mbar_init(xchg_bar(b), 32 * C::kEpiWarps);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc<512>(smem_u32(tmem_slot));
  __syncthreads();
  if (warp == 0) {  // inclusive scan of prefix[1..E]
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
        if (p.mode == kGateUp) {
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
          const int x = kb * C::kBK;
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
        if constexpr (!FP8) {
          const int buf = acc_it & 1, use = acc_it >> 1;
          if (!mbar_wait(tempty_bar(buf), (use & 1) ^ 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
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
            for (int k = 0; k < C::kMmaPerStage; ++k)
              umma_f16(d, da + 2 * k, db + 2 * k, C::kIdesc, (kb | k) != 0);
            umma_commit(empty_bar(s));
          }
          if (!ok) break;
          umma_commit(tfull_bar(buf));
          ++acc_it;
        } else {
          for (int kb = 0; kb < num_kb; ++kb, ++it, ++acc_it) {
            const int buf = acc_it & 1, use = acc_it >> 1;
            const int s = it % kStages, round = it / kStages;
            if (!mbar_wait(tempty_bar(buf), (use & 1) ^ 1) ||
                !mbar_wait(full_bar(s), round & 1)) {
              set_err(p.err, GBMOE_ERR_TIMEOUT);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + buf * kBN;
            const uint64_t da = umma_desc_sw128(sA + s * kAStage);
            const uint64_t db = umma_desc_sw128(sB + s * kBStage);
#pragma unroll
            for (int k = 0; k < C::kMmaPerStage; ++k)
              umma_f8(d, da + 2 * k, db + 2 * k, C::kIdesc, k != 0);
            umma_commit(empty_bar(s));
            umma_commit(tfull_bar(buf));
          }
        }
      }
      // every MMA issued above has finished before TMEM is released
      umma_commit(done_bar);
      mbar_wait(done_bar, 0, 100000000ull);
    }
  } else {
    // ============================= epilogue =============================
    const int ew = warp - 2;             // epilogue warp index
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int half = ew >> 2;            // fp8: column half of this warp
    const int row_in_tile = q * 32 + lane;
    const uint32_t t_lane = (uint32_t)(q * 32) << 16;
    int acc_it = 0, tile_no = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++tile_no) {
      int e, mt, nt;
      decode_tile(prefix, E, p.n_tiles, tile, e, mt, nt);
      const int r = mt * kBM + row_in_tile;  // row within the expert
      const bool valid = r < rcnt[e];
      const int arow = rbase[e] + r;         // row of A / H
      if constexpr (!FP8) {
        const int buf = acc_it & 1, use = acc_it >> 1;
        if (!mbar_wait(tfull_bar(buf), use & 1)) {
          set_err(p.err, GBMOE_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + t_lane + buf * kBN;
        if (p.mode == kGateUp) {
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
              const float h0 = silu_f(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
              const float h1 = silu_f(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
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
              w = p.topk_w[pair];
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
        if (lane == 0) mbar_arrive(tempty_bar(buf));
        ++acc_it;
      } else {
        // ---- fp8: promote each K block's partial sums with its scales
        float acc[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
        // scale rows of the weight tile: gate/up blocks (kGateUp) or the two
        // 128-row blocks of the 256-column tile (kDown); one per column half
        const int b_blk_rows = p.b_rows / 128;
        int blk0, blk1;
        if (p.mode == kGateUp) {
          blk0 = nt;
          blk1 = p.N / 128 + nt;
        } else {
          blk0 = blk1 = nt * 2 + half;
          if (blk0 >= b_blk_rows) blk0 = blk1 = b_blk_rows - 1;  // columns masked
        }
        const float *bs0 = p.b_scales + ((size_t)e * b_blk_rows + blk0) * num_kb;
        const float *bs1 = p.b_scales + ((size_t)e * b_blk_rows + blk1) * num_kb;
        const float *as = p.a_scales + (size_t)arow * num_kb;
        auto ld_scales = [&](int kb, float &sa, float &sb0, float &sb1) {
          if (kb < num_kb) {
            sa = valid ? as[kb] : 0.0f;
            sb0 = bs0[kb];
            sb1 = bs1[kb];
          }
        };
        float sa0 = 0.f, sg0 = 0.f, su0 = 0.f, sa1 = 0.f, sg1 = 0.f, su1 = 0.f;
        ld_scales(0, sa0, sg0, su0);
        ld_scales(1, sa1, sg1, su1);
        for (int kb = 0; kb < num_kb; ++kb, ++acc_it) {
          float sa2 = 0.f, sg2 = 0.f, su2 = 0.f;
          ld_scales(kb + 2, sa2, sg2, su2);
          const int buf = acc_it & 1, use = acc_it >> 1;
          if (!mbar_wait(tfull_bar(buf), use & 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tb = tmem_base + t_lane + buf * kBN;
          const float f0 = sa0 * sg0, f1 = sa0 * su0;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            // kGateUp: chunks 0,1 gate columns half*64 + [0,64), chunks 2,3 up
            // columns 128 + half*64 + [0,64).  kDown: columns half*128 + 32c.
            const uint32_t col = p.mode == kGateUp
                                     ? (uint32_t)((c >> 1) * 128 + half * 64 + (c & 1) * 32)
                                     : (uint32_t)(half * 128 + c * 32);
            uint32_t v[32];
            tmem_ld32(tb + col, v);
            tmem_ld_wait();
            const float f = (p.mode == kGateUp && c >= 2) ? f1 : f0;
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[c * 32 + i] = fmaf(f, __uint_as_float(v[i]), acc[c * 32 + i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(buf));
          sa0 = sa1; sg0 = sg1; su0 = su1;
          sa1 = sa2; sg1 = sg2; su1 = su2;
        }
        if (!ok) break;
        if (p.mode == kGateUp) {
          // h = silu(gate) * up on this thread's 64 columns, then e4m3 with
          // one scale per 128-wide group (this tile's columns, both halves)
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            acc[i] = silu_f(acc[i]) * acc[64 + i];
            amax = fmaxf(amax, fabsf(acc[i]));
          }
          const int xb = tile_no & 1;
          amax_x[(xb * 2 + half) * 128 + row_in_tile] = amax;
          mbar_arrive(xchg_bar(xb));
          if (!mbar_wait(xchg_bar(xb), (tile_no >> 1) & 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
          amax = fmaxf(amax, amax_x[(xb * 2 + (half ^ 1)) * 128 + row_in_tile]);
          const float s = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
          if (valid) {
            uint8_t *hrow = static_cast<uint8_t *>(p.out) + (size_t)arow * p.N + nt * 128 + half * 64;
            uint4 *dst = reinterpret_cast<uint4 *>(hrow);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w4[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int i0 = v * 16 + j * 4;
                w4[j] = e4m3x4(__fdiv_rn(acc[i0], s), __fdiv_rn(acc[i0 + 1], s),
                               __fdiv_rn(acc[i0 + 2], s), __fdiv_rn(acc[i0 + 3], s));
              }
              dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            if (half == 0) p.out_scales[(size_t)arow * (p.N / 128) + nt] = s;
          }
        } else {
          size_t orow = 0;
          float w = 1.0f;
          if (valid) {
            if (p.sorted) {
              const int pair = p.sorted[arow];
              orow = (size_t)pair;
              w = p.topk_w[pair];
            } else {
              orow = (size_t)arow;
            }
          }
          const int col0 = nt * kBN + half * 128;
          if (valid && col0 < p.K) {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + orow * p.K + col0);
#pragma unroll
            for (int v = 0; v < 16; ++v)
              dst[v] = make_uint4(pack_bf16x2(w * acc[8 * v], w * acc[8 * v + 1]),
                                  pack_bf16x2(w * acc[8 * v + 2], w * acc[8 * v + 3]),
                                  pack_bf16x2(w * acc[8 * v + 4], w * acc[8 * v + 5]),
                                  pack_bf16x2(w * acc[8 * v + 6], w * acc[8 * v + 7]));
          }
        }
      }
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

bool resolve_encode() {
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode != nullptr;
}

template <bool FP8>
cudaError_t launch_impl(const GroupedGemmArgs &a, int num_sms, cudaStream_t s) {
  using C = Cfg<FP8>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t st = cudaFuncSetAttribute(grouped_gemm_kernel<FP8>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          kSmemBytes);
    if (st != cudaSuccess) return st;
    attr_set = true;
  }
  const bool gate_up = a.mode == kGateUp;
  const int Kd = gate_up ? a.K : a.N;          // contraction length
  const int b_rows = gate_up ? 2 * a.N : a.K;  // rows of B per expert
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, a.A, C::kElemBytes, (uint64_t)Kd, (uint64_t)a.a_rows,
                      C::kBK, kBM) ||
      !encode_tmap_2d(&tmB, a.B, C::kElemBytes, (uint64_t)Kd,
                      (uint64_t)a.E * b_rows, C::kBK, 128))
    return cudaErrorInvalidValue;
  KParams p;
  p.mode = a.mode;
  p.offsets = a.offsets;
  p.counts = a.counts;
  p.E = a.E;
  p.T = a.T;
  p.N = a.N;
  p.K = a.K;
  p.n_tiles = gate_up ? a.N / 128 : (a.K + kBN - 1) / kBN;
  p.num_kb = Kd / C::kBK;
  p.a_rows = (int)a.a_rows;
  p.b_rows = b_rows;
  p.out = a.out;
  p.out_scales = a.out_scales;
  p.a_scales = a.A_scales;
  p.b_scales = a.B_scales;
  p.sorted = a.sorted_pair_ids;
  p.topk_w = a.topk_weights;
  p.err = a.err;
  // upper bound on the tiles: every expert may end with a partial m-tile
  long long mtiles = a.offsets ? (a.a_rows + kBM - 1) / kBM + a.E
                               : (long long)a.E * ((a.T + kBM - 1) / kBM);
  long long tiles = mtiles * p.n_tiles;
  int grid = (int)(tiles < num_sms ? tiles : num_sms);
  if (grid < 1) grid = 1;
  grouped_gemm_kernel<FP8><<<grid, C::kThreads, kSmemBytes, s>>>(tmA, tmB, p);
  return cudaGetLastError();
}

}  // namespace

bool encode_tmap_2d(CUtensorMap *map, const void *base, int elem_bytes,
                    uint64_t cols, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows) {
  if (!resolve_encode()) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_grouped_gemm(const GroupedGemmArgs &a, int num_sms,
                                cudaStream_t s) {
  return a.fp8 ? launch_impl<true>(a, num_sms, s) : launch_impl<false>(a, num_sms, s);
}

}  // namespace gbmoe

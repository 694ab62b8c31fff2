// gemm_fp8.cu -- the two expert GEMMs with e4m3 operands and fp32 block
// scales (1 x 128 along K for the rows of A, 128 x 128 for the weights), on
// tcgen05.mma kind::f8f6f4 with the fp32 scale promotion done by the
// epilogue warps.
//
// Both scales change every 128 elements of K, so a K block's products cannot
// be accumulated across blocks inside the tensor core.  Each K block (4 MMAs
// of K 32) is accumulated alone into one of two 256-column TMEM buffers; 8
// epilogue warps then add it into fp32 registers,
//     acc += (s_a[row, kb] * s_w[blk, kb]) * partial,
// while the tensor core fills the other buffer.  Each epilogue thread owns one
// row and 128 columns (4 lane quarters x 2 column halves cover the 128 x 256
// tile: for gate/up the gate and up columns of 64 outputs), so the promotion
// is 64 packed FFMA2 per thread per K block, in 16-column TMEM loads; at 352
// threads (with the output warp below) a thread has 168 registers, enough
// for its 128 accumulators.  The
// per-row scales of a K block travel with the operand tiles: the producer
// loads them by TMA from the group-major scale array (one contiguous run of
// rows per K block) into the stage's shared memory; the weight-block scales
// of a tile (two rows of K blocks) are staged in shared memory once per tile.
//
// gate/up ends with h = silu(gate) * up and the e4m3 requantisation of h in
// 128-wide groups (one scale per row and n-tile, from the maximum of the two
// half-rows that two warps hold); down ends with the
// router weight and bf16 stores into the (token, slot) rows, or unweighted
// into the row itself in the BatchedExperts format (row groups from the
// device counts, e*T + [0, count)) (the ordered
// top-k reduce is a pass of its own after this kernel: added to this
// epilogue it stalled the per-K-block pipeline, 1.8 -> 4.3 ms on the
// DeepSeek-V3-shaped prefill).
//
// The epilogue keeps its accumulators in registers, so the tensor core can
// run only two K blocks into the next tile while the epilogue finishes the
// current one.  Down tiles are short (K = N, 16 K blocks for N = 2048), and
// writing 128 scattered output rows per tile from the epilogue stalled the
// next tile's MMAs for about a third of the tile's time.  So the epilogue
// only puts its rows into a shared-memory stage of the whole tile (down:
// bf16 rows times the router weight; gate/up: h in fp32 and each half-row's
// maximum) and an output warp stores them (gate/up: after the scales and the
// e4m3 codes) during the next tile; the stage costs the operand ring one of
// four stages.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "per_device.h"

namespace gbmoe {

namespace {

using namespace gemm;

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kBK = kBKB;                       // e4m3 elements per stage row
constexpr int kMmaPerStage = kBK / 32;          // kind::f8f6f4 has K = 32
constexpr uint32_t kIdesc = umma_idesc(kBM, kBN, kFmtE4M3);
constexpr int kMaxKB = 128;                     // K up to 16384
constexpr int kASBox = kBM + 4;                 // row scales per K block (rows from a 4-aligned start)
constexpr int kASStage = 640;                   // bytes per ring slot (528 used)
static_assert(kASStage % 128 == 0, "a TMA destination in shared memory is 128-byte aligned");
constexpr int kASStages = 8;                    // row-scale ring, deeper than the operand ring

// a staged output row: 128 fp32 h values (gate/up) or 256 bf16 (down), plus
// 16 bytes of padding so that 32 rows' 16-byte accesses spread over the banks
constexpr int kTileRow = 528;

// Shared-memory layout per mode: three operand stages, then the stage of the
// whole output tile that the output warp drains while the epilogue moves on
// to the next tile (gate/up: h in fp32 with the two half-rows' maxima and
// the rows' 1/scale; down: the bf16 rows with their pair ids).
// Barriers: full[S], empty[S], tfull[2], tempty[2], done, bsc[2], (2 unused),
// as_full[8], as_empty[8], stg_full, stg_empty.
template <int MODE>
struct Layout {
  static constexpr bool kDown = MODE == kDownMode;
  static constexpr int S = 3;
  static constexpr int threads = 64 + kEpiThreads + 32;  // + the output warp
  static constexpr int offA = 0;
  static constexpr int offB = offA + S * kAStage;
  static constexpr int offAS = offB + S * kBStage;
  static constexpr int offBar = offAS + kASStages * kASStage;
  static constexpr int nbars = 2 * S + 2 + 2 + 1 + 2 + 2 + 2 * kASStages + 2;
  static constexpr int offTmem = offBar + 8 * nbars;
  static constexpr int offBsc = offTmem + 16;                      // [2 bufs][2][kMaxKB] f32
  static constexpr int offRowMax = offBsc + 2 * 2 * kMaxKB * 4;    // gate/up: [2 halves][128], [128] 1/s
  static constexpr int offStg = (offRowMax + (kDown ? 0 : 3 * 128 * 4) + 127) / 128 * 128;
  static constexpr int offStgPair = offStg + kBM * kTileRow;
  static constexpr int offPrefix = offStgPair + (kDown ? kBM * 4 : 0);
  static constexpr int offRBase = offPrefix + (kMaxE + 1) * 4;
  static constexpr int offRCnt = offRBase + kMaxE * 4;
  static constexpr int used = offRCnt + kMaxE * 4;
  static constexpr int smem = used + 1024;
  static_assert(smem <= 232448, "shared memory");
};

struct KParams {
  const int32_t *offsets;   // Standard: expert e owns rows [offsets[e], offsets[e+1])
  const int32_t *counts;    // Batched (offsets NULL): rows [e*T, e*T + min(counts[e], T))
  int T;
  int E, N, K;
  int n_tiles;
  int num_kb;
  int b_rows;               // rows of B per expert (2N or K)
  void *out;
  float *out_scales;        // gate/up: H scales (N/128, scale_ld)
  int64_t scale_ld;
  const float *b_scales;    // (E, b_rows/128, num_kb)
  const int32_t *sorted;    // down: output row of each row of A (NULL: the row itself)
  const float *topk_w;
  int32_t *err;
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}


// acc[0..8) += f * v[0..16) (as 8 float2) with packed fp32x2 FMAs
__device__ __forceinline__ void promote8(float2 *acc, const uint32_t (&v)[16], float f) {
  const float2 f2 = make_float2(f, f);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    acc[j] = __ffma2_rn(make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), f2, acc[j]);
}

template <int MODE, int ACT>
__global__ void __launch_bounds__(Layout<MODE>::threads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmAS,
                            const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw_u32);

  using L = Layout<MODE>;
  constexpr int S = L::S;
  const uint32_t sA = base + L::offA;
  const uint32_t sB = base + L::offB;
  const uint32_t sAS = base + L::offAS;
  const uint32_t bar0 = base + L::offBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * S + 4);
  auto bsc_bar = [&](int b) { return bar0 + 8u * (2 * S + 5 + b); };
  auto as_full_bar = [&](int s) { return bar0 + 8u * (2 * S + 9 + s); };
  auto as_empty_bar = [&](int s) { return bar0 + 8u * (2 * S + 9 + kASStages + s); };
  const uint32_t stg_full_bar = bar0 + 8u * (2 * S + 9 + 2 * kASStages);
  const uint32_t stg_empty_bar = stg_full_bar + 8u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + L::offTmem);
  const float *as_smem = reinterpret_cast<const float *>(sbase + L::offAS);
  float *bsc_smem = reinterpret_cast<float *>(sbase + L::offBsc);
  float *rowmax = reinterpret_cast<float *>(sbase + L::offRowMax);
  uint8_t *stg = sbase + L::offStg;
  int *stg_pair = reinterpret_cast<int *>(sbase + L::offStgPair);
  int *prefix = reinterpret_cast<int *>(sbase + L::offPrefix);
  int *rbase = reinterpret_cast<int *>(sbase + L::offRBase);
  int *rcnt = reinterpret_cast<int *>(sbase + L::offRCnt);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  tile_table_fill(p.offsets, p.counts, E, p.T, p.n_tiles, prefix, rbase, rcnt, p.err);
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < kASStages; ++s) {
      mbar_init(as_full_bar(s), 1);
      mbar_init(as_empty_bar(s), kEpiWarps);  // every epilogue warp has read its scale
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps);
      mbar_init(bsc_bar(b), kEpiThreads);
    }
    mbar_init(done_bar, 1);
    mbar_init(stg_full_bar, kEpiWarps);  // every epilogue warp staged its rows
    mbar_init(stg_empty_bar, 1);         // the store / quant warp drained the stage
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmAS);
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
      int last_round[S], last_as_round[kASStages];
#pragma unroll
      for (int s = 0; s < S; ++s) last_round[s] = -1;
#pragma unroll
      for (int s = 0; s < kASStages; ++s) last_as_round[s] = -1;
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
          const int s = it % S, round = it / S;
          const int s8 = it % kASStages, round8 = it / kASStages;
          if (!mbar_wait(empty_bar(s), (round & 1) ^ 1) ||
              !mbar_wait(as_empty_bar(s8), (round8 & 1) ^ 1)) {
            set_err(p.err, GBMOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), kAStage + kBStage);
          const int x = kb * kBK;
          tma_load_2d(sA + s * kAStage, &tmA, full_bar(s), x, a_row);
          tma_load_2d(sB + s * kBStage, &tmB, full_bar(s), x, b_row0);
          tma_load_2d(sB + s * kBStage + kBStage / 2, &tmB, full_bar(s), x, b_row1);
          last_round[s] = round;
          // row scales of K block kb for rows [a_row & ~3, +132): the start
          // is rounded down to 4 floats (16 bytes) as TMA requires
          mbar_arrive_expect_tx(as_full_bar(s8), kASBox * 4);
          tma_load_2d(sAS + s8 * kASStage, &tmAS, as_full_bar(s8), a_row & ~3, kb);
          last_as_round[s8] = round8;
        }
      }
      // copies still in flight land before the CTA can leave
#pragma unroll
      for (int s = 0; s < S; ++s)
        if (last_round[s] >= 0) mbar_wait(full_bar(s), last_round[s] & 1, 100000000ull);
#pragma unroll
      for (int s = 0; s < kASStages; ++s)
        if (last_as_round[s] >= 0) mbar_wait(as_full_bar(s), last_as_round[s] & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer =============================
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int buf = it & 1, use = it >> 1;
          const int s = it % S, round = it / S;
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
          for (int k = 0; k < kMmaPerStage; ++k)
            umma_f8(d, da + 2 * k, db + 2 * k, kIdesc, k != 0);
          umma_commit(empty_bar(s));
          umma_commit(tfull_bar(buf));
        }
      }
      umma_commit(done_bar);
      mbar_wait(done_bar, 0, 100000000ull);
    }
  } else if (MODE == kDownMode && warp == 2 + kEpiWarps) {
    // ========================= down-output stores =======================
    // Each staged row goes out as one 512-byte store (32 lanes x 16 B) to
    // its (token, slot) row; the stage is handed back once read.
    int tile_no = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tile_no) {
      int e, mt, nt;
      decode_tile(prefix, E, p.n_tiles, tile, e, mt, nt);
      if (!mbar_wait(stg_full_bar, tile_no & 1)) {
        set_err(p.err, GBMOE_ERR_TIMEOUT);
        break;
      }
      const int col = nt * kBN + lane * 8;
      const bool in_k = col < p.K;
      uint16_t *ycol = static_cast<uint16_t *>(p.out) + col;
#pragma unroll 8
      for (int r = 0; r < kBM; ++r) {
        const int pr = stg_pair[r];
        if (pr >= 0 && in_k) {
          const uint4 v = *reinterpret_cast<const uint4 *>(stg + r * kTileRow + lane * 16);
          *reinterpret_cast<uint4 *>(ycol + (size_t)pr * p.K) = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(stg_empty_bar);
    }
  } else if (MODE == kGateUpMode && warp == 2 + kEpiWarps) {
    // ===================== h requantisation and stores ==================
    // A staged row holds h of the tile's 128 outputs in fp32 and the maxima
    // of its two halves.  Lane l first turns rows l, l + 32, ... into their
    // scales (s = max / 448) and 1/s; then every row's codes go out as one
    // 128-byte store, lane l coding outputs [4l, 4l + 4).
    const float *hst = reinterpret_cast<const float *>(stg);
    float *rinv = rowmax + 2 * 128;  // [128] 1 / scale of each staged row
    int tile_no = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tile_no) {
      int e, mt, nt;
      decode_tile(prefix, E, p.n_tiles, tile, e, mt, nt);
      if (!mbar_wait(stg_full_bar, tile_no & 1)) {
        set_err(p.err, GBMOE_ERR_TIMEOUT);
        break;
      }
      const int rows = min(rcnt[e] - mt * kBM, kBM);
      const int arow0 = rbase[e] + mt * kBM;
      // one row's scale per lane: the maximum of its two halves' maxima
      for (int r = lane; r < rows; r += 32) {
        const float amax = fmaxf(rowmax[r], rowmax[128 + r]);
        const float sc = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
        rinv[r] = __frcp_rn(sc);  // codes of h * (1 / s)
        p.out_scales[(size_t)nt * p.scale_ld + arow0 + r] = sc;
      }
      __syncwarp();
      uint8_t *hrow = static_cast<uint8_t *>(p.out) + (size_t)arow0 * p.N + nt * 128;
#pragma unroll 4
      for (int r = 0; r < rows; ++r) {
        const float4 h = *reinterpret_cast<const float4 *>(hst + r * (kTileRow / 4) + lane * 4);
        const float inv_sc = rinv[r];
        reinterpret_cast<uint32_t *>(hrow + (size_t)r * p.N)[lane] =
            e4m3x4(h.x * inv_sc, h.y * inv_sc, h.z * inv_sc, h.w * inv_sc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(stg_empty_bar);
    }
  } else {
    // ============================= epilogue =============================
    const int ew = warp - 2;           // 0..7
    const int q = warp & 3;            // TMEM lane quarter of this warp
    const int hh = ew >> 2;            // column half of this warp
    const int etid = ew * 32 + lane;   // 0..255
    const int row_in_tile = q * 32 + lane;
    const uint32_t t_lane = (uint32_t)(q * 32) << 16;
    const int b_blk_rows = p.b_rows / 128;
    // The weight-block scales of a tile, [0] gate (or the first 128
    // columns), [1] up (or the second 128 columns), for every K block:
    // 2 * num_kb <= 256 values, one per epilogue thread.  Each thread loads
    // its value of the next tile while the current one runs and stores it
    // into the other half of the double buffer at the tile's end, so a tile
    // starts with its scales in shared memory.
    auto tile_scale = [&](int te, int tnt) -> float {
      if (etid >= 2 * num_kb) return 0.0f;
      const int h = etid / num_kb, kb = etid - h * num_kb;
      int blk = MODE == kGateUpMode ? (h == 0 ? tnt : p.N / 128 + tnt) : tnt * 2 + h;
      if (blk >= b_blk_rows) blk = b_blk_rows - 1;  // columns past K: masked
      return __ldg(p.b_scales + ((size_t)te * b_blk_rows + blk) * num_kb + kb);
    };
    auto put_scale = [&](int tno, float v) {
      if (etid < 2 * num_kb) {
        const int h = etid / num_kb, kb = etid - h * num_kb;
        bsc_smem[(tno & 1) * 2 * kMaxKB + h * kMaxKB + kb] = v;
      }
      mbar_arrive(bsc_bar(tno & 1));
    };
    // down: the output row (pair) of this thread's row and its router weight
    auto row_pair = [&](int te, int tmt) -> int {
      if (tmt * kBM + row_in_tile >= rcnt[te]) return -1;
      const int r = rbase[te] + tmt * kBM + row_in_tile;
      return p.sorted ? __ldg(p.sorted + r) : r;
    };
    // a tile is decoded once, as the next tile of the previous iteration
    int ce = 0, cmt = 0, cnt = 0;
    int cur_pair = 0;
    float cur_wgt = 1.0f;
    if (blockIdx.x < total) {
      decode_tile(prefix, E, p.n_tiles, blockIdx.x, ce, cmt, cnt);
      put_scale(0, tile_scale(ce, cnt));
      if (MODE == kDownMode) {
        cur_pair = row_pair(ce, cmt);
        cur_wgt = cur_pair >= 0 && p.topk_w ? __ldg(p.topk_w + cur_pair) : 1.0f;
      }
    }
    int it = 0, tile_no = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++tile_no) {
      const int e = ce, mt = cmt, nt = cnt;
      const int a_row = rbase[e] + mt * kBM;
      const int r = mt * kBM + row_in_tile;
      const bool valid = r < rcnt[e];
      const int as_idx = (a_row & 3) + row_in_tile;
      // the next tile: its decode, its weight-block scale (stored at this
      // tile's end) and, for down, its row's pair (the weight of that pair
      // is loaded halfway through this tile's K loop)
      const bool has_next = tile + (int)gridDim.x < total;
      int ne = 0, nmt = 0, nnt = 0;
      if (has_next) decode_tile(prefix, E, p.n_tiles, tile + gridDim.x, ne, nmt, nnt);
      const float next_scale = has_next ? tile_scale(ne, nnt) : 0.0f;
      const int pair = cur_pair;
      const float wgt = cur_wgt;
      const int nxt_pair = MODE == kDownMode && has_next ? row_pair(ne, nmt) : -1;
      float nxt_wgt = 1.0f;

      const int tb = tile_no & 1;
      const float *bsc = bsc_smem + tb * 2 * kMaxKB;
      if (!mbar_wait(bsc_bar(tb), (tile_no >> 1) & 1)) {
        set_err(p.err, GBMOE_ERR_TIMEOUT);
        break;
      }
      const float *bs_g = bsc;                     // gate
      const float *bs_u = bsc + kMaxKB;            // up
      const float *bs_d = bsc + hh * kMaxKB;       // down: this half's weight block

      // gate/up: [0, 32) the gate of columns [64 hh, 64 hh + 64), [32, 64)
      // their up; down: columns [128 hh, 128 hh + 128)
      float2 acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);

      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        if (MODE == kDownMode && kb == num_kb / 2 && nxt_pair >= 0 && p.topk_w)
          nxt_wgt = __ldg(p.topk_w + nxt_pair);
        const int buf = it & 1, use = it >> 1;
        const int s8 = it % kASStages, round8 = it / kASStages;
        if (!mbar_wait(as_full_bar(s8), round8 & 1)) {
          set_err(p.err, GBMOE_ERR_TIMEOUT);
          ok = false;
          break;
        }
        const float sa = as_smem[s8 * (kASStage / 4) + as_idx];
        __syncwarp();
        if (lane == 0) mbar_arrive(as_empty_bar(s8));
        if (!mbar_wait(tfull_bar(buf), use & 1)) {
          set_err(p.err, GBMOE_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbuf = tmem_base + t_lane + buf * kBN;
        uint32_t v[16];
        if (MODE == kGateUpMode) {
          const float fg = sa * bs_g[kb], fu = sa * bs_u[kb];
          const uint32_t cg = tbuf + hh * 64, cu = tbuf + 128 + hh * 64;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_ld16(cg + 16 * c, v);
            tmem_ld_wait();
            promote8(acc + 8 * c, v, fg);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_ld16(cu + 16 * c, v);
            tmem_ld_wait();
            promote8(acc + 32 + 8 * c, v, fu);
          }
        } else {
          const float f = sa * bs_d[kb];
          const uint32_t c0 = tbuf + hh * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            tmem_ld16(c0 + 16 * c, v);
            tmem_ld_wait();
            promote8(acc + 8 * c, v, f);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
      }
      if (!ok) break;

      if (MODE == kGateUpMode) {
        // h on this thread's 64 columns into the tile's stage; the quant
        // warp requantises and stores it while this warp starts the next tile
        if (!mbar_wait(stg_empty_bar, (tile_no & 1) ^ 1)) {
          set_err(p.err, GBMOE_ERR_TIMEOUT);
          break;
        }
        float4 *dst = reinterpret_cast<float4 *>(stg + row_in_tile * kTileRow + hh * 256);
        float amax = 0.0f;
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const float2 g0 = acc[2 * v], g1 = acc[2 * v + 1];
          const float2 u0 = acc[32 + 2 * v], u1 = acc[32 + 2 * v + 1];
          const float4 h = make_float4(gate_act_fast<ACT>(g0.x) * u0.x, gate_act_fast<ACT>(g0.y) * u0.y,
                                       gate_act_fast<ACT>(g1.x) * u1.x, gate_act_fast<ACT>(g1.y) * u1.y);
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w))));
          dst[v] = h;
        }
        rowmax[hh * 128 + row_in_tile] = amax;  // this half-row's maximum
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_full_bar);
      } else {
        // This thread's 128 columns (256 bytes of bf16) of its row go into
        // the tile's stage; the store warp writes them out while this warp
        // starts on the next tile.
        if (!mbar_wait(stg_empty_bar, (tile_no & 1) ^ 1)) {
          set_err(p.err, GBMOE_ERR_TIMEOUT);
          break;
        }
        if (nt * kBN + hh * 128 < p.K) {  // uniform over the warp
          uint4 *dst = reinterpret_cast<uint4 *>(stg + row_in_tile * kTileRow + hh * 256);
#pragma unroll
          for (int v = 0; v < 16; ++v)
            dst[v] = make_uint4(pack_bf16x2(wgt * acc[4 * v].x, wgt * acc[4 * v].y),
                                pack_bf16x2(wgt * acc[4 * v + 1].x, wgt * acc[4 * v + 1].y),
                                pack_bf16x2(wgt * acc[4 * v + 2].x, wgt * acc[4 * v + 2].y),
                                pack_bf16x2(wgt * acc[4 * v + 3].x, wgt * acc[4 * v + 3].y));
        }
        if (hh == 0) stg_pair[row_in_tile] = valid ? pair : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_full_bar);
      }
      if (has_next) put_scale(tile_no + 1, next_scale);
      cur_pair = nxt_pair;
      cur_wgt = nxt_wgt;
      ce = ne;
      cmt = nmt;
      cnt = nnt;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<512>(tmem_base);
}

template <int MODE, int ACT>
cudaError_t launch_fp8(const GroupedGemmArgs &a, int num_sms, cudaStream_t s) {
  static PerDeviceInt smem_set;
  cudaError_t st = set_smem_once(smem_set, grouped_gemm_fp8_kernel<MODE, ACT>, Layout<MODE>::smem);
  if (st != cudaSuccess) return st;
  const bool gate_up = MODE == kGateUpMode;
  const int Kd = gate_up ? a.K : a.N;
  const int b_rows = gate_up ? 2 * a.N : a.K;
  const int num_kb = Kd / kBK;
  if (num_kb > kMaxKB || a.scale_ld % 4 != 0 || a.scale_ld < a.a_rows)
    return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB, tmAS;
  if (!encode_tmap_2d(&tmA, a.A, kTmapU8, (uint64_t)Kd, (uint64_t)a.a_rows, (uint64_t)Kd,
                      kBK, kBM, true) ||
      !encode_tmap_2d(&tmB, a.B, kTmapU8, (uint64_t)Kd, (uint64_t)a.E * b_rows, (uint64_t)Kd,
                      kBK, 128, true) ||
      !encode_tmap_2d(&tmAS, a.A_scales, kTmapF32, (uint64_t)a.scale_ld, (uint64_t)num_kb,
                      (uint64_t)a.scale_ld * 4, kASBox, 1, false))
    return cudaErrorInvalidValue;
  KParams p;
  p.offsets = a.offsets;
  p.counts = a.counts;
  p.T = a.T;
  p.E = a.E;
  p.N = a.N;
  p.K = a.K;
  p.n_tiles = gate_up ? a.N / 128 : (a.K + kBN - 1) / kBN;
  p.num_kb = num_kb;
  p.b_rows = b_rows;
  p.out = a.out;
  p.out_scales = a.out_scales;
  p.scale_ld = a.scale_ld;
  p.b_scales = a.B_scales;
  p.sorted = a.sorted_pair_ids;
  p.topk_w = a.topk_weights;
  p.err = a.err;
  long long tiles = ((a.a_rows + kBM - 1) / kBM + a.E) * (long long)p.n_tiles;
  int grid = (int)(tiles < num_sms ? tiles : num_sms);
  if (grid < 1) grid = 1;
  grouped_gemm_fp8_kernel<MODE, ACT><<<grid, Layout<MODE>::threads, Layout<MODE>::smem, s>>>(tmA, tmB, tmAS, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_fp8(const GroupedGemmArgs &a, int num_sms,
                                    cudaStream_t s) {
  if (a.mode == kDown) return launch_fp8<kDownMode, kActSilu>(a, num_sms, s);
  return a.act == GBMOE_ACT_GELU ? launch_fp8<kGateUpMode, kActGelu>(a, num_sms, s)
                                 : launch_fp8<kGateUpMode, kActSilu>(a, num_sms, s);
}

}  // namespace gbmoe

// gemm.cu - MXFP8 block-scaled GEMMs on the 5th-generation tensor cores (tcgen05,
// kind::mxf8f6f4 with UE8M0 scales), dense and grouped over MoE token segments.
//
// Method: "End-to-End MXFP8 RL on Blackwell" (verl blog post), section "The pipeline":
// the format paragraph (Blackwell tensor cores take the 32-element block scales as
// operands of the MMA instruction) and the learner paragraph (forward, data-gradient
// and weight-gradient GEMMs per linear layer); expert GEMMs of Qwen3-30B-A3B: section
// "A held-out workload, and end to end", Table 4.
//
// Kernel design: persistent CTAs, warp-specialised, 320 threads.
//   warp 0      TMA producer: per 128-wide K stage, tiled loads of the A and B tiles with
//               the 128-byte swizzle and of the stage's scale tiles; the whole warp runs
//               the loop and one elected lane issues.
//   warp 1      allocates TMEM; its elected lane copies the stage's scale tiles into TMEM
//               (tcgen05.cp 32x128b.warpx4: a 512-byte swizzled tile lands as 4 TMEM
//               columns, byte k of each column = K block k) and issues the stage's
//               block-scaled MMAs (K = 32 each) into the FP32 accumulator in TMEM.
//   warps 2-9   epilogue, two warps per TMEM lane quarter: tcgen05.ld of the accumulator,
//               FP32 -> BF16 (or FP32), stores through shared memory with TMA.
// Two kernels share this layout:
//   mxfp8_gemm_2sm_kernel  clusters of two CTAs on two SMs compute 256 x BN tiles with
//                          tcgen05.mma.cta_group::2: BN = 256, 192 (two accumulators) or
//                          384 (two N = 192 MMAs sharing the A stage); the dense GEMMs
//                          with N > 128 and the grouped GEMMs for up to 256 experts.
//   mxfp8_gemm_kernel      one CTA per SM, 128 x 256 or 128 x 128 tiles; everything else.
// No load is multicast across a cluster: every CTA loads its own operand tiles.
// Shared-memory stages are recycled through full/empty mbarriers; the accumulator
// through acc_full/acc_empty, so the producer already streams the next tile's operands
// while the epilogue drains the current one. Each stage has its own TMEM scale slot,
// so a slot is only rewritten after the MMAs that read it have completed (the stage's
// empty barrier, armed by tcgen05.commit, precedes its refill).
// Every wait is bounded: past the limit the CTA latches MXFP8_ERR_TIMEOUT, all roles
// leave their loops, outstanding copies and MMAs are waited for, TMEM is freed.
// A partial last wave of 2SM tiles runs as half-width tiles, or, for deep reductions with
// a caller-owned workspace (mxfp8_gemm_ws), as split-K pieces in a separate kernel
// instance. Every kernel is launched with programmatic stream serialization: it sets up,
// then waits for the previous kernel before touching global memory.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"
#include "mxfp8.h"

namespace mxfp8 {
namespace {

constexpr int BM = 128;           // accumulator rows = TMEM lanes
constexpr int BK = 128;           // K elements (bytes) per pipeline stage
constexpr int kEpiWarps = 8;      // two per TMEM lane quarter, each half of the columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
// Split-K of a 384-wide kernel's last wave: each tile of it runs as this many K pieces.
constexpr int kSplitK = 3;
constexpr int kMaxExperts = 1024;

enum Mode : int { kDense = 0, kGroupRows = 1, kGroupWgrad = 2 };

template <int BN>
struct Cfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kSfbTiles = BN / 128;
  static constexpr int kSfbBytes = kSfbTiles * 512;
  // shared memory carve-up (offsets from a 1024-byte aligned base)
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kStages * 512;
  static constexpr int kOffBar = kOffSfb + kStages * kSfbBytes;
  static constexpr int kNumBars = 2 * kStages + 3;  // full, empty, acc_full, acc_empty, done
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // epilogue staging: one 32-row x 64-byte box (2 KB) per epilogue warp, 1024-aligned
  static constexpr int kStageBoxBytes = 32 * 64;
  static constexpr int kOffOut = (kOffMisc + 64 + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = kOffOut + kEpiWarps * kStageBoxBytes + 1024;  // + slack
  // TMEM columns: accumulator, then per-stage scale slots
  static constexpr int kSfaCol = BN;
  static constexpr int kSfbCol = BN + 4 * kStages;
  static constexpr int kColsUsed = kSfbCol + (BN / 32) * kStages;
  static constexpr int kTmemCols = kColsUsed <= 256 ? 256 : 512;
  static_assert(kColsUsed <= 512, "TMEM overflow");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory overflow");
};

struct Params {
  const uint8_t* sA;
  const uint8_t* sB;
  void* C;
  int64_t M, N;          // output rows / cols of one problem
  int64_t K;             // reduction length (dense / grouped rows)
  int out_fp32;
  const int32_t* offsets;
  int E;
  int64_t total_rows;
  int64_t sb_item_bytes; // grouped rows: bytes of one expert's B scale block
  int64_t num_tiles;     // dense: all tiles; grouped: upper bound
  int num_m_tiles, num_n_tiles;
  int band;              // dense: M tiles (2SM kernel: pairs of M tiles) per raster band
  int* status;
  uint64_t wait_ns;      // pipeline waits give up after this (MXFP8_ERR_TIMEOUT)
  uint64_t drain_ns;     // waits for work already in flight, on the way out (never shorter)
  // dense 2SM kernel: the pair tiles from this index on run as two half-width tiles, or (the
  // split-K kernel instance) as kSplitK pieces that each take a range of K of the whole tile
  int64_t split_from = INT64_MAX;
  uint4* ws = nullptr;           // split-K: FP32 partials of pieces 0 .. kSplitK - 2
  uint32_t* ws_flags = nullptr;  // split-K: one arrival counter per (tile, CTA rank, epilogue
                                 // warp); zero between launches
};

// Everything a role needs to know about one output tile.
struct Tile {
  int64_t m0, n0;        // output tile origin within its problem
  int rows_valid, cols_valid;
  int64_t a_row;         // TMA row coordinate of A
  int64_t k_origin;      // TMA K coordinate of the first stage
  int nk;                // K stages
  int last_blocks;       // valid 32-blocks in the last stage (1..4)
  int b_z;               // expert index for the 3-D B map (grouped rows)
  int64_t sfa_tile0;     // scale tile index of (row tile, stage 0) in sA
  int64_t sfa_kstride;   // tiles between consecutive stages (1)
  const uint8_t* sfb_base;
  int64_t sfb_row_tiles_stride;  // tiles between consecutive 128-row B tiles
  int c_z;               // the problem's index in the output map (expert for wgrad)
  bool live;
};

struct SegShared {
  int32_t off[kMaxExperts + 1];
  int32_t tile_base[kMaxExperts + 1];
  int16_t order[kMaxExperts];  // experts by decreasing token count (ties: lower index first)
  int ok;
};

__device__ int find_seg(const SegShared& s, int E, int64_t t) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.tile_base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int BN, int kMode>
__device__ Tile make_tile(const Params& p, const SegShared* seg, int64_t id) {
  Tile t;
  t.live = false;
  const int64_t n_kt_dense = (p.K + BK - 1) / BK;
  if (kMode == kDense) {
    if (id >= p.num_tiles) return t;
    // banded raster: bands of p.band M tiles sweep across N, M fastest within a band, so
    // that concurrent CTAs share operand tiles in L2 (the band width is chosen on the host)
    // 32-bit arithmetic: the host keeps tile counts below 2^31
    const uint32_t uid = static_cast<uint32_t>(id);
    const uint32_t GM = static_cast<uint32_t>(p.band);
    const uint32_t band = GM * static_cast<uint32_t>(p.num_n_tiles);
    const uint32_t g = uid / band, r = uid - g * band;
    const uint32_t first_m = g * GM;
    const uint32_t gm = (static_cast<uint32_t>(p.num_m_tiles) - first_m) < GM
                            ? (static_cast<uint32_t>(p.num_m_tiles) - first_m) : GM;
    const uint32_t nt32 = r / gm;
    const int64_t mt = first_m + (r - nt32 * gm);
    const int64_t nt = nt32;
    t.m0 = mt * BM;
    t.n0 = nt * BN;
    t.rows_valid = static_cast<int>((p.M - t.m0) < BM ? (p.M - t.m0) : BM);
    t.cols_valid = static_cast<int>((p.N - t.n0) < BN ? (p.N - t.n0) : BN);
    t.a_row = t.m0;
    t.k_origin = 0;
    t.nk = static_cast<int>(n_kt_dense);
    t.last_blocks = static_cast<int>(((p.K - (n_kt_dense - 1) * BK) + 31) / 32);
    t.b_z = 0;
    t.sfa_tile0 = mt * n_kt_dense;
    t.sfa_kstride = 1;
    t.sfb_base = p.sB + nt * (BN / 128) * n_kt_dense * 512;
    t.sfb_row_tiles_stride = n_kt_dense;
    t.c_z = 0;
    t.live = true;
    return t;
  }
  if (kMode == kGroupRows) {
    const int64_t n_tiles = static_cast<int64_t>(seg->tile_base[p.E]) * p.num_n_tiles;
    if (!seg->ok || id >= n_tiles) return t;
    const uint32_t uid = static_cast<uint32_t>(id), nnt = static_cast<uint32_t>(p.num_n_tiles);
    const int64_t row_tile = uid / nnt;
    const int64_t nt = uid - static_cast<uint32_t>(row_tile) * nnt;
    const int e = find_seg(*seg, p.E, row_tile);
    const int64_t i = row_tile - seg->tile_base[e];
    t.m0 = seg->off[e] + i * BM;
    t.n0 = nt * BN;
    const int64_t left = seg->off[e + 1] - t.m0;
    t.rows_valid = static_cast<int>(left < BM ? left : BM);
    t.cols_valid = static_cast<int>((p.N - t.n0) < BN ? (p.N - t.n0) : BN);
    t.a_row = t.m0;
    t.k_origin = 0;
    t.nk = static_cast<int>(n_kt_dense);
    t.last_blocks = static_cast<int>(((p.K - (n_kt_dense - 1) * BK) + 31) / 32);
    t.b_z = e;
    t.sfa_tile0 = row_tile * n_kt_dense;
    t.sfa_kstride = 1;
    t.sfb_base = p.sB + e * p.sb_item_bytes + nt * (BN / 128) * n_kt_dense * 512;
    t.sfb_row_tiles_stride = n_kt_dense;
    t.c_z = 0;
    t.live = true;
    return t;
  }
  // grouped weight gradient: problem e is [M = N_out] x [N = K_out], reduced over the
  // tokens of segment e
  // Experts are visited heaviest first, so the CTAs' static round robin over the tiles
  // spreads the long reductions evenly (longest-processing-time-first order).
  const int64_t per = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
  if (!seg->ok || id >= per * p.E) return t;
  const uint32_t uid = static_cast<uint32_t>(id), uper = static_cast<uint32_t>(per);
  const uint32_t nnt = static_cast<uint32_t>(p.num_n_tiles);
  const uint32_t ei = uid / uper, r = uid - ei * uper;
  const int e = seg->order[ei];
  const uint32_t mt32 = r / nnt;
  const int64_t mt = mt32, nt = r - mt32 * nnt;
  const int64_t cnt = seg->off[e + 1] - seg->off[e];
  const int64_t nk = (cnt + BK - 1) / BK;
  t.m0 = mt * BM;
  t.n0 = nt * BN;
  t.rows_valid = static_cast<int>((p.M - t.m0) < BM ? (p.M - t.m0) : BM);
  t.cols_valid = static_cast<int>((p.N - t.n0) < BN ? (p.N - t.n0) : BN);
  t.a_row = t.m0;
  t.k_origin = seg->off[e];
  t.nk = static_cast<int>(nk);
  t.last_blocks = nk ? static_cast<int>((cnt - (nk - 1) * BK) / 32) : 0;
  t.b_z = 0;
  const int64_t n_rt_a = (p.M + 127) / 128, n_rt_b = (p.N + 127) / 128;
  const int64_t tb = seg->tile_base[e];
  t.sfa_tile0 = n_rt_a * tb + mt * nk;
  t.sfa_kstride = 1;
  t.sfb_base = p.sB + (n_rt_b * tb + nt * (BN / 128) * nk) * 512;
  t.sfb_row_tiles_stride = nk;
  t.c_z = e;
  t.live = true;
  return t;
}

// Waits, with the drain limit, for every stage use in [consumed, issued) to land on its full
// barrier, then for the last arrival of the MMA issuer's commits on each empty barrier
// (consumed uses) and on each accumulator barrier (`commits` of them, kAcc buffers). A
// parity wait is exact here: no barrier has run more than one phase past the one waited for.
template <int kStages, int kAcc>
__device__ void drain_stages(uint64_t* full, uint64_t* empty, uint64_t* acc_full,
                             uint32_t issued, uint32_t consumed, uint32_t commits,
                             uint64_t limit_ns) {
  for (uint32_t i = consumed; i < issued; ++i)
    mbar_wait_timed(&full[i % kStages], (i / kStages) & 1, limit_ns);
  for (uint32_t i = consumed > kStages ? consumed - kStages : 0; i < consumed; ++i)
    mbar_wait_timed(&empty[i % kStages], (i / kStages) & 1, limit_ns);
  for (uint32_t k = commits > kAcc ? commits - kAcc : 0; k < commits; ++k)
    mbar_wait_timed(&acc_full[k % kAcc], (k / kAcc) & 1, limit_ns);
}

template <int BN, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
mxfp8_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                  const __grid_constant__ CUtensorMap map_b,
                  const __grid_constant__ CUtensorMap map_c, const Params p) {
  using C = Cfg<BN>;
  // persistent tile loop: CTAs stride over the tile list
  const int64_t first_id = blockIdx.x;
  const int64_t id_step = gridDim.x;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* acc_full = bars + 2 * C::kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* mma_done = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  // drain records: [0] stage uses issued by the producer, [1] stage uses consumed by the
  // MMA issuer, [2] accumulator commits, [3] the producer's tail completed
  volatile uint32_t* rec = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 8);
  __shared__ SegShared seg_storage;
  SegShared* seg = (kMode == kDense) ? nullptr : &seg_storage;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
    tma_prefetch_desc(&map_c);
  }
  if (kMode != kDense) grid_dependency_wait();  // the offsets may come from the previous kernel
  if (kMode != kDense) {
    // segment table: offsets checked (0-based, non-decreasing, 32-aligned, ending at
    // total_rows) and prefix sums of ceil(count / 128)
    const int E = p.E;
    if (threadIdx.x == 0) seg->ok = 1;
    __syncthreads();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) seg->off[i] = p.offsets[i];
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
      const int32_t lo = seg->off[i], hi = seg->off[i + 1];
      if (hi < lo || (lo & 31) || (hi & 31)) seg->ok = 0;
    }
    if (threadIdx.x == 0 &&
        (seg->off[0] != 0 || static_cast<int64_t>(seg->off[E]) != p.total_rows))
      seg->ok = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
      int32_t acc = 0;
      for (int e = 0; e < E; ++e) {
        seg->tile_base[e] = acc;
        const int32_t cnt = seg->off[e + 1] - seg->off[e];
        acc += cnt > 0 ? (cnt + 127) / 128 : 0;
      }
      seg->tile_base[E] = acc;
      if (!seg->ok && blockIdx.x == 0) latch_error(p.status, MXFP8_ERR_BAD_OFFSETS);
    }
    if (kMode == kGroupWgrad) {
      // rank of expert e = experts with more tokens, or as many and a lower index
      for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t ce = seg->off[e + 1] - seg->off[e];
        int rank = 0;
        for (int f = 0; f < E; ++f) {
          const int32_t cf = seg->off[f + 1] - seg->off[f];
          rank += (cf > ce) || (cf == ce && f < e);
        }
        seg->order[rank] = static_cast<int16_t>(e);
      }
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (kMode == kDense) grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    // whole warp in the loop (warp-uniform addresses), one elected lane issues the copies
    const bool issuer = elect_one();
    uint32_t it = 0;
    bool ok = true;
    for (int64_t id = first_id; ok; id += id_step) {
      const Tile t = make_tile<BN, kMode>(p, seg, id);
      if (!t.live) break;
      int n_sfb = 0;
      for (int h = 0; h < C::kSfbTiles; ++h) n_sfb += (t.n0 + 128 * h < p.N);
      const uint32_t bytes = C::kABytes + C::kBBytes + 512 + 512 * n_sfb;
      for (int kb = 0; kb < t.nk; ++kb, ++it) {
        const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1;
        if (!warp_wait(&empty[s], ph ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
        if (issuer) {
          mbar_arrive_expect_tx(&full[s], bytes);
          const int32_t kx = static_cast<int32_t>(t.k_origin + static_cast<int64_t>(kb) * BK);
          tma_load_2d(smem + C::kOffA + s * C::kABytes, &map_a, kx,
                      static_cast<int32_t>(t.a_row), &full[s]);
          if (kMode == kGroupRows)
            tma_load_3d(smem + C::kOffB + s * C::kBBytes, &map_b, kx, static_cast<int32_t>(t.n0),
                        t.b_z, &full[s]);
          else
            tma_load_2d(smem + C::kOffB + s * C::kBBytes, &map_b, kx, static_cast<int32_t>(t.n0),
                        &full[s]);
          bulk_load(smem + C::kOffSfa + s * 512, p.sA + (t.sfa_tile0 + kb) * 512, 512, &full[s]);
          for (int h = 0; h < n_sfb; ++h)
            bulk_load(smem + C::kOffSfb + s * C::kSfbBytes + h * 512,
                      t.sfb_base + (h * t.sfb_row_tiles_stride + kb) * 512, 512, &full[s]);
        }
        __syncwarp();
      }
    }
    if (!ok && issuer) {
      *abort_flag = 1;
      latch_error(p.status, MXFP8_ERR_TIMEOUT);
    }
    if (issuer) rec[0] = it;  // the copies still in flight are waited for on the way out
    // Producer tail: the MMA issuer's release of the last stage uses must have arrived on
    // their empty barriers before the CTA exits. Waiting here overlaps the epilogue's last
    // tile; after an abort the drain below does it instead.
    bool tail_ok = ok;
    for (uint32_t i = it > C::kStages ? it - C::kStages : 0; tail_ok && i < it; ++i)
      tail_ok = warp_wait(&empty[i % C::kStages], (i / C::kStages) & 1, abort_flag, p.wait_ns);
    if (issuer) rec[3] = tail_ok ? 1u : 0u;
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop, so that every descriptor and address is warp-uniform
    // (uniform registers); one elected lane issues the tensor-core instructions. The loop
    // is kept short: descriptors are built once and advanced by adding 16-byte units to
    // their start-address field (shared addresses stay below 2^18, so no carry leaves it).
    const bool issuer = elect_one();
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    const uint64_t a_desc0 = smem_desc(smem_u32(smem + C::kOffA), 16, 1024, 2);
    const uint64_t b_desc0 = smem_desc(smem_u32(smem + C::kOffB), 16, 1024, 2);
    const uint64_t sfa_desc0 = smem_desc(smem_u32(smem + C::kOffSfa), 0, 128, 0);
    const uint64_t sfb_desc0 = smem_desc(smem_u32(smem + C::kOffSfb), 0, 128, 0);
    constexpr uint32_t kId0 = mxf8_idesc(BM, BN, 0, 0), kId1 = mxf8_idesc(BM, BN, 1, 1);
    constexpr uint32_t kId2 = mxf8_idesc(BM, BN, 2, 2), kId3 = mxf8_idesc(BM, BN, 3, 3);
    for (int64_t id = first_id; ok; id += id_step) {
      const Tile t = make_tile<BN, kMode>(p, seg, id);
      if (!t.live) break;
      if (t.nk == 0) continue;
      if (!warp_wait(acc_empty, (acc_it & 1) ^ 1, abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < t.nk; ++kb, ++it) {
        const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1;
        if (!warp_wait(&full[s], ph, abort_flag, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sfa_t = tmem + C::kSfaCol + 4 * s;
        const uint32_t sfb_t = tmem + C::kSfbCol + (BN / 32) * s;
        const uint64_t ad = a_desc0 + s * (C::kABytes / 16);
        const uint64_t bd = b_desc0 + s * (C::kBBytes / 16);
        const uint32_t acc0 = kb > 0 ? 1u : 0u;
        if (issuer) {
          tmem_cp_32x128b_x4(sfa_t, sfa_desc0 + s * (512 >> 4));
#pragma unroll
          for (int h = 0; h < C::kSfbTiles; ++h)
            tmem_cp_32x128b_x4(sfb_t + 4 * h, sfb_desc0 + (s * C::kSfbBytes + h * 512) / 16);
          if (kb != t.nk - 1 || t.last_blocks == 4) {  // K step k starts 32 bytes further
            mma_mxf8(tmem, ad, bd, kId0, sfa_t, sfb_t, acc0);
            mma_mxf8(tmem, ad + 2, bd + 2, kId1, sfa_t, sfb_t, 1u);
            mma_mxf8(tmem, ad + 4, bd + 4, kId2, sfa_t, sfb_t, 1u);
            mma_mxf8(tmem, ad + 6, bd + 6, kId3, sfa_t, sfb_t, 1u);
          } else {
            for (int k = 0; k < t.last_blocks; ++k)
              mma_mxf8(tmem, ad + 2 * k, bd + 2 * k, mxf8_idesc(BM, BN, k, k), sfa_t, sfb_t,
                       (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (issuer) mma_commit(acc_full);
      __syncwarp();
      ++acc_it;
    }
    if (!ok && issuer) {
      *abort_flag = 1;
      latch_error(p.status, MXFP8_ERR_TIMEOUT);
    }
    // all issued tensor-core work must be finished before TMEM is released
    if (issuer) {
      rec[1] = it;
      rec[2] = acc_it;
      mma_commit(mma_done);
      mbar_wait_timed(mma_done, 0, p.drain_ns);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the BN columns
    constexpr int kChunks = BN / 64;   // 32-column chunks per warp
    uint8_t* box = smem + C::kOffOut + (warp - 2) * C::kStageBoxBytes;
    uint32_t acc_it = 0;
    bool ok = true;
    for (int64_t id = first_id; ok; id += id_step) {
      const Tile t = make_tile<BN, kMode>(p, seg, id);
      if (!t.live) break;
      if (t.nk > 0) {
        // one lane waits, the warp follows its verdict (keeps the warp converged)
        int got = 0;
        if (lane == 0) got = mbar_wait_bounded(acc_full, acc_it & 1, abort_flag, p.wait_ns);
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) { ok = false; break; }
        tc_fence_after();
      }
      // The whole accumulator slice of this warp (32 rows x BN/2 columns) goes to
      // registers first, and TMEM is handed back to the MMA issuer before any store, so
      // the next tile's MMAs overlap this tile's conversion and stores.
      uint32_t v[kChunks][32];
      __syncwarp();
      if (t.nk > 0) {
        const uint32_t base = tmem + (static_cast<uint32_t>(32 * q) << 16) + half * kChunks * 32;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tmem_ld_32x32b_x32(base + 32 * c, v[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(acc_empty);
        ++acc_it;
      } else {
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[c][i] = 0;
      }
      // Stores leave through shared memory: each 64-byte column group of the warp's 32 rows
      // is written into the warp's staging box (16-byte chunks XOR-swizzled as the tensor
      // map's 64-byte swizzle expects) and sent with one TMA store, clipped at the matrix
      // edge. Segments are 32-row aligned, so a box never crosses into another expert.
      if (32 * q < t.rows_valid) {
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const int c = half * kChunks + u;
          if (32 * c >= t.cols_valid) continue;
#pragma unroll
          for (int g = 0; g < (p.out_fp32 ? 2 : 1); ++g) {
            const int col = 32 * c + 16 * g;  // first column of this group
            if (col >= t.cols_valid) continue;
            uint4 w[4];
            if (p.out_fp32) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                w[j] = make_uint4(v[u][16 * g + 4 * j], v[u][16 * g + 4 * j + 1],
                                  v[u][16 * g + 4 * j + 2], v[u][16 * g + 4 * j + 3]);
            } else {
              uint32_t b[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                b[i] = cvt_bf16x2(__uint_as_float(v[u][2 * i + 1]), __uint_as_float(v[u][2 * i]));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                w[j] = make_uint4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
            }
            if (lane == 0) bulk_wait_read_all();  // the box is free again
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(box + lane * 64 + 16 * (j ^ ((lane >> 1) & 3))) = w[j];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&map_c, box, static_cast<int32_t>(t.n0 + col),
                           static_cast<int32_t>(t.m0 + 32 * q), t.c_z);
              bulk_commit_group();
            }
          }
        }
      }
    }
    // Before the CTA exits its stores must have finished reading its shared memory; the
    // kernel's completion makes their global writes visible to later work.
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    if (!ok && lane == 0) {
      *abort_flag = 1;
      latch_error(p.status, MXFP8_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  // Drain, after an abort: whatever stopped the loops, nothing this CTA started may still be
  // writing its shared memory or arriving on its barriers when it exits. Loads of the stage
  // uses that the MMA issuer never consumed complete by themselves (every byte of a stage
  // comes from this CTA's own copies); the last arrivals of the MMA issuer's commits are
  // waited for too. These waits have their own limit, never shorter than the pipeline's.
  // Without an abort every use was consumed, the producer's tail has seen the last releases
  // and the epilogue every accumulator commit, so there is nothing left to wait for.
  if (threadIdx.x == 0 && !(rec[3] && !*abort_flag && rec[0] == rec[1]))
    drain_stages<C::kStages, 1>(full, empty, acc_full, rec[0], rec[1], rec[2], p.drain_ns);
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------- dense GEMM on CTA pairs (2SM)
//
// A cluster of two CTAs on two SMs computes 256 x BN output tiles with
// tcgen05.mma.cta_group::2 (M = 256). Each CTA stages, per 128-wide K stage, its own 128
// rows of A, its own BN/2 rows of the B tile (B is split between the pair), the scale tile
// of its A rows and the two 128-row scale tiles of B that cover the tile's BN columns.
// Against one-SM 128 x 256 tiles this halves the B bytes each SM stages and reads, and the
// scale copies per flop. Every copy of either CTA completes on the leader's `full` barrier;
// the leader's tcgen05.commit frees a stage in both CTAs and hands an accumulator to both
// epilogues, whose 16 warps return it on the leader's `acc_empty`.
//
// BN = 256 keeps one accumulator (256 of the 512 TMEM columns, the rest hold the scale
// slots). BN = 192 fits two accumulators and seven stages' scale slots, so the next
// tile's MMAs run while the epilogue drains the previous one. A 192-column tile starts
// either on a 128-row scale tile or 64 rows into one. Both scale tiles are always copied
// to the slot's 4-aligned columns; in the second case the MMA's B-scale address is two
// columns further on, where the scales of the tile's B rows 0-31 are.
constexpr int kMaxDuoExperts = 256;  // grouped GEMMs on the 2SM kernel (segment table size)

// Expert segments of a grouped 2SM GEMM, rebuilt by every CTA from the offsets.
struct DuoSeg {
  int32_t off[kMaxDuoExperts + 1];
  int32_t tile_base[kMaxDuoExperts + 1];  // prefix sums of ceil(count / 128)
  int32_t pair_base[kMaxDuoExperts + 1];  // prefix sums of ceil(ceil(count / 128) / 2)
  int16_t order[kMaxDuoExperts];          // experts by decreasing count (ties: lower index)
  int ok;
};

// BN = 384 (dense, BF16 output): each K step issues two N = 192 MMAs that share the A
// stage, into accumulator columns [0, 192) and [192, 384); each CTA stages two 96-row B
// boxes (rows 96c.. and 192 + 96c.. of the pair tile). Fewer staged bytes and scale copies
// per FLOP than a 256-wide tile, and fewer tiles to hand over per launch.
template <int BN, int kMode = kDense>
struct Duo {
  static constexpr bool kGrouped = kMode != kDense;
  static constexpr bool kWide = BN == 384;
  static_assert(!kWide || kMode != kGroupWgrad, "384-wide tiles: dense and grouped rows");
  static constexpr int kMmaN = kWide ? 192 : BN;       // N of one MMA instruction
  static constexpr int kBoxRows = kWide ? 96 : BN / 2; // B rows per TMA box
  static constexpr int kAcc = BN == 192 ? 2 : 1;       // accumulator buffers
  static constexpr int kStages = BN == 256 ? 6 : (kWide ? 5 : (kGrouped ? 6 : 7));
  static constexpr int kABytes = BM * BK;              // own 128 A rows
  static constexpr int kBBytes = (BN / 2) * BK;        // own half of the B tile
  static constexpr int kSfaBytes = 512;
  static constexpr int kSfbTiles = kWide ? 3 : 2;      // 128-row scale tiles of B per stage
  static constexpr int kSfbBytes = 512 * kSfbTiles;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  // a 384-wide kernel's half tile stages its first B box only
  static constexpr int kHalfStageBytes = kWide ? kStageBytes - kBoxRows * BK : kStageBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
  static constexpr int kOffBar = kOffSfb + kStages * kSfbBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kAcc + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // epilogue staging: one 32-row box per epilogue warp, 1024-aligned; 64-byte rows, or
  // 32-byte rows for 384-wide tiles (which leave less shared memory)
  static constexpr int kBoxRowBytes = kWide ? 32 : 64;
  static constexpr int kStageBoxBytes = 32 * kBoxRowBytes;
  static constexpr int kOffOut = (kOffMisc + 64 + 1023) / 1024 * 1024;
  static constexpr int kOffSeg = kOffOut + kEpiWarps * kStageBoxBytes;
  static constexpr int kSmemBytes =
      kOffSeg + (kGrouped ? static_cast<int>(sizeof(DuoSeg)) : 0) + 1024;
  static constexpr int kSfaCol = kAcc * BN;            // TMEM: accumulators, then scales
  static constexpr int kSfbSlot = 4 * kSfbTiles;       // columns per B scale slot
  static constexpr int kSfbCol = kSfaCol + 4 * kStages;
  static constexpr int kTmemCols = 512;
  static constexpr int kAccEmptyCount = 2 * kEpiWarps;  // epilogue warps of both CTAs
  static_assert(kSfbCol + kSfbSlot * kStages <= kTmemCols, "TMEM overflow");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory overflow");
  static_assert(kBBytes % 1024 == 0, "B stages must keep the 1024-byte swizzle alignment");
};

struct DuoTile {
  int64_t m0 = 0;        // this CTA's first output row (within its problem)
  int64_t n0 = 0;        // the pair tile's first output column
  int64_t mt = 0;        // this CTA's 128-row tile index (its A rows and their scales)
  int64_t sfb_tile = 0;  // first 128-row scale tile of B the pair tile touches
  int sfb_shift = 0;     // 0, or 2 when the tile starts 64 rows into that scale tile
  int rows_valid = 0, cols_valid = 0;
  bool live = false;
  int nk = 0;                  // K stages of this tile (0: an empty expert's zero tile)
  int last_blocks = 0;         // 32-blocks of K in the last stage
  int64_t k_origin = 0;        // TMA K coordinate of the first stage (grouped wgrad)
  int64_t sfa_idx = 0;         // grouped: flat scale tile index of this CTA's A rows, stage 0
  int64_t sfb_idx0 = 0, sfb_idx1 = 0, sfb_idx2 = 0;  // grouped: the B scale tiles, stage 0
  int b_z = 0, c_z = 0;        // expert index for the B (grouped rows) and C (wgrad) maps
  int width = 0;               // output columns of the tile: BN, or BN / 2 for a half tile
  int kb0 = 0;                 // first K stage of a split-K piece (else 0)
  int piece = -1;              // split-K piece index, -1 for a whole tile or a half tile
  int slot = 0;                // split-K: the tile's index among the split tiles
};

// Dense pair tiles. Work item `pid` below p.split_from is pair tile pid. From there on the
// items share pair tiles, in one of two ways:
// - two items per tile, each taking half of its columns (256 x BN/2);
// - kSplitK items per tile, each taking a range of its K stages (the split-K instance).
// The host puts the split at the last, partial wave of clusters when the pieces fit in one
// wave, so that wave takes a fraction as long.
// The work-item arithmetic is 32-bit: the host checks that the pair tiles and items of a
// launch stay below 2^31, and 64-bit divisions (emulated in software) cost every role a
// visible delay before its first tile.
template <int BN, bool kSplit>
__device__ __forceinline__ DuoTile duo_tile(const Params& p, int64_t item, uint32_t crank) {
  DuoTile t;
  const uint32_t n_pm = static_cast<uint32_t>((p.num_m_tiles + 1) / 2);
  uint32_t pid = static_cast<uint32_t>(item);
  int half = -1;  // -1: the whole tile; 0 / 1: its left / right half
  if (item >= p.split_from) {
    const uint32_t r = static_cast<uint32_t>(item - p.split_from);
    if constexpr (kSplit) {
      const uint32_t slot = r / static_cast<uint32_t>(kSplitK);
      pid = static_cast<uint32_t>(p.split_from) + slot;
      t.piece = static_cast<int>(r - slot * static_cast<uint32_t>(kSplitK));
      t.slot = static_cast<int>(slot);
    } else {
      pid = static_cast<uint32_t>(p.split_from) + r / 2;
      half = static_cast<int>(r & 1);
    }
  }
  t.live = pid < n_pm * static_cast<uint32_t>(p.num_n_tiles);
  if (!t.live) return t;
  const uint32_t GP = static_cast<uint32_t>(p.band);  // bands of GP pair rows sweep across
  const uint32_t band = GP * static_cast<uint32_t>(p.num_n_tiles);  // N, pair rows fastest
  const uint32_t bi = pid / band, r = pid - bi * band;
  const uint32_t first = bi * GP;
  const uint32_t gp = (n_pm - first) < GP ? (n_pm - first) : GP;
  const uint32_t nt = r / gp;
  const int64_t pm = first + (r - nt * gp);
  t.mt = 2 * pm + crank;
  t.m0 = t.mt * BM;
  t.width = half < 0 ? BN : BN / 2;
  t.n0 = nt * BN + (half > 0 ? BN / 2 : 0);
  t.sfb_tile = t.n0 / 128;
  t.sfb_shift = static_cast<int>((t.n0 % 128) / 32);
  const int64_t left = p.M - t.m0;
  t.rows_valid = static_cast<int>(left <= 0 ? 0 : (left < BM ? left : BM));
  const int64_t cols = p.N - t.n0;
  t.cols_valid = static_cast<int>(cols <= 0 ? 0 : (cols < t.width ? cols : t.width));
  return t;
}

// Grouped pair tiles.
//  kGroupRows: expert e's token rows are cut into 128-row tiles; a pair takes two adjacent
//  tiles of one expert (the second may lie past the segment: computed, never stored) and
//  one BN-column tile of N, against expert e's weight (B map z = e).
//  kGroupWgrad: problem e is dW[e] = dY_e^T X_e, [M = N_out] x [N = K_out], reduced over
//  expert e's tokens; experts are visited heaviest first.
// Scale tiles are addressed by flat index in the grouped layouts (512 bytes each).
template <int BN, int kMode>
__device__ DuoTile duo_tile_grouped(const Params& p, const DuoSeg* seg, int64_t pid,
                                    uint32_t crank) {
  DuoTile t;
  t.live = false;
  if (!seg->ok) return t;
  const int E = p.E;
  const int64_t n_kt = (p.K + BK - 1) / BK;
  const int64_t n_rt_b = (p.N + 127) / 128;
  if (kMode == kGroupRows) {
    const int64_t total = static_cast<int64_t>(seg->pair_base[E]) * p.num_n_tiles;
    if (pid >= total) return t;
    const uint32_t upid = static_cast<uint32_t>(pid), nnt = static_cast<uint32_t>(p.num_n_tiles);
    const uint32_t rp32 = upid / nnt;
    const int64_t rp = rp32, nt = upid - rp32 * nnt;
    int lo = 0, hi = E - 1;  // expert owning pair row rp
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seg->pair_base[mid] <= rp) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int64_t j = 2 * (rp - seg->pair_base[e]) + crank;  // row tile within the expert
    t.m0 = seg->off[e] + j * BM;
    const int64_t left = seg->off[e + 1] - t.m0;
    t.rows_valid = static_cast<int>(left <= 0 ? 0 : (left < BM ? left : BM));
    t.n0 = nt * BN;
    t.cols_valid = static_cast<int>((p.N - t.n0) < BN ? (p.N - t.n0) : BN);
    t.nk = static_cast<int>(n_kt);
    t.last_blocks = static_cast<int>(((p.K - (n_kt - 1) * BK) + 31) / 32);
    t.k_origin = 0;
    // indices of tiles that do not exist (an odd last row tile, the second B scale tile
    // past N) fall back to a tile that does: their rows and columns are never stored
    const int64_t rt = seg->tile_base[e + 1] - seg->tile_base[e];
    t.sfa_idx = (seg->tile_base[e] + (j < rt ? j : rt - 1)) * n_kt;
    const int64_t h = t.n0 / 128;
    t.sfb_idx0 = (e * n_rt_b + h) * n_kt;
    t.sfb_idx1 = h + 1 < n_rt_b ? t.sfb_idx0 + n_kt : t.sfb_idx0;
    t.sfb_idx2 = h + 2 < n_rt_b ? t.sfb_idx0 + 2 * n_kt : t.sfb_idx1;  // 384-wide tiles
    t.b_z = e;
    t.c_z = 0;
  } else {
    const int64_t n_pm = ((p.M + 127) / 128 + 1) / 2;
    const int64_t per = n_pm * p.num_n_tiles;
    if (pid >= per * E) return t;
    const uint32_t upid = static_cast<uint32_t>(pid), uper = static_cast<uint32_t>(per);
    const uint32_t nnt = static_cast<uint32_t>(p.num_n_tiles);
    const uint32_t ei = upid / uper, r = upid - ei * uper;
    const int e = seg->order[ei];
    const uint32_t pm32 = r / nnt;
    const int64_t pm = pm32, nt = r - pm32 * nnt;
    const int64_t cnt = seg->off[e + 1] - seg->off[e];
    const int64_t nk = (cnt + BK - 1) / BK;
    const int64_t mt = 2 * pm + crank;
    t.m0 = mt * BM;
    const int64_t left = p.M - t.m0;
    t.rows_valid = static_cast<int>(left <= 0 ? 0 : (left < BM ? left : BM));
    t.n0 = nt * BN;
    t.cols_valid = static_cast<int>((p.N - t.n0) < BN ? (p.N - t.n0) : BN);
    t.nk = static_cast<int>(nk);
    t.last_blocks = nk ? static_cast<int>((cnt - (nk - 1) * BK) / 32) : 0;
    t.k_origin = seg->off[e];
    const int64_t tb = seg->tile_base[e];
    const int64_t n_rt_a = (p.M + 127) / 128;
    t.sfa_idx = n_rt_a * tb + (mt < n_rt_a ? mt : n_rt_a - 1) * nk;
    const int64_t h = t.n0 / 128;
    t.sfb_idx0 = n_rt_b * tb + h * nk;
    t.sfb_idx1 = h + 1 < n_rt_b ? t.sfb_idx0 + nk : t.sfb_idx0;
    t.b_z = 0;
    t.c_z = e;
  }
  t.mt = 0;
  t.sfb_tile = 0;
  t.sfb_shift = static_cast<int>((t.n0 % 128) / 32);
  t.width = BN;
  t.live = true;
  return t;
}

template <int BN, int kMode, bool kSplit = false>
__device__ __forceinline__ DuoTile duo_tile_of(const Params& p, const DuoSeg* seg, int64_t pid,
                                               uint32_t crank) {
  if constexpr (kMode == kDense) {
    DuoTile t = duo_tile<BN, kSplit>(p, pid, crank);
    t.nk = static_cast<int>((p.K + BK - 1) / BK);
    t.last_blocks = static_cast<int>(((p.K - (t.nk - 1) * BK) + 31) / 32);
    t.c_z = 0;
    if (kSplit && t.piece >= 0) {  // split-K: stages [nk * i / S, nk * (i + 1) / S)
      constexpr int S = kSplitK;
      const int nk = t.nk;
      t.kb0 = nk * t.piece / S;
      t.nk = nk * (t.piece + 1) / S - t.kb0;
      if (t.piece != S - 1) t.last_blocks = 4;  // only the last piece holds the ragged stage
    }
    return t;
  } else {
    return duo_tile_grouped<BN, kMode>(p, seg, pid, crank);
  }
}

// Bytes one CTA stages for its stage use number `use` (the producer's running count):
// found by walking the CTA's tiles again. Only the drain after an abort needs it.
template <int BN, int kMode, bool kSplit>
__device__ uint32_t duo_use_bytes(const Params& p, const DuoSeg* seg, int64_t first_id,
                                  int64_t id_step, uint32_t crank, uint32_t use) {
  using D = Duo<BN, kMode>;
  if constexpr (D::kHalfStageBytes == D::kStageBytes) {
    return D::kStageBytes;
  } else {
    uint32_t at = 0;
    for (int64_t id = first_id;; id += id_step) {
      const DuoTile t = duo_tile_of<BN, kMode, kSplit>(p, seg, id, crank);
      if (!t.live) break;
      if (use < at + static_cast<uint32_t>(t.nk))
        return t.width == BN ? D::kStageBytes : D::kHalfStageBytes;
      at += static_cast<uint32_t>(t.nk);
    }
    return D::kStageBytes;
  }
}

// kSplit: the dense kernel whose last wave runs as split-K pieces (a separate instance, so
// that the split code costs the other launches nothing).
template <int BN, int kMode, bool kSplit = false>
__global__ void __launch_bounds__(kThreads, 1)
mxfp8_gemm_2sm_kernel(const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b,
                      const __grid_constant__ CUtensorMap map_sfa,
                      const __grid_constant__ CUtensorMap map_sfb,
                      const __grid_constant__ CUtensorMap map_c, const Params p) {
  using D = Duo<BN, kMode>;
  constexpr int kStages = D::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + D::kOffBar);
  uint64_t* full = bars;                    // the leader's count both CTAs' bytes
  uint64_t* empty = bars + kStages;         // armed in both CTAs by the leader's commit
  uint64_t* acc_full = bars + 2 * kStages;  // [kAcc], armed in both CTAs
  uint64_t* acc_empty = acc_full + D::kAcc; // [kAcc], the leader's are used
  uint64_t* mma_done = acc_empty + D::kAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + D::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + D::kOffMisc + 4);
  // drain records, in both CTAs: [0] / [1] stage uses issued by the producer of CTA 0 / 1,
  // [2] stage uses consumed by the MMA issuer, [3] accumulator commits; [4] this CTA's
  // producer tail completed
  volatile uint32_t* rec = reinterpret_cast<volatile uint32_t*>(smem + D::kOffMisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int64_t first_id = blockIdx.x >> 1;
  const int64_t id_step = gridDim.x >> 1;
  DuoSeg* seg = D::kGrouped ? reinterpret_cast<DuoSeg*>(smem + D::kOffSeg) : nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < D::kAcc; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], D::kAccEmptyCount);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
    tma_prefetch_desc(&map_sfa);
    tma_prefetch_desc(&map_sfb);
    tma_prefetch_desc(&map_c);
  }
  if constexpr (D::kGrouped) grid_dependency_wait();  // the offsets may come from the previous kernel
  if constexpr (D::kGrouped) {
    // segment table: offsets checked (0-based, non-decreasing, 32-aligned, ending at
    // total_rows), prefix sums, and the heaviest-first expert order
    const int E = p.E;
    if (threadIdx.x == 0) seg->ok = 1;
    __syncthreads();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) seg->off[i] = p.offsets[i];
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
      const int32_t lo = seg->off[i], hi = seg->off[i + 1];
      if (hi < lo || (lo & 31) || (hi & 31)) seg->ok = 0;
    }
    if (threadIdx.x == 0 &&
        (seg->off[0] != 0 || static_cast<int64_t>(seg->off[E]) != p.total_rows))
      seg->ok = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
      int32_t tiles = 0, pairs = 0;
      for (int e = 0; e < E; ++e) {
        seg->tile_base[e] = tiles;
        seg->pair_base[e] = pairs;
        const int32_t cnt = seg->off[e + 1] - seg->off[e];
        const int32_t rt = cnt > 0 ? (cnt + 127) / 128 : 0;
        tiles += rt;
        pairs += (rt + 1) / 2;
      }
      seg->tile_base[E] = tiles;
      seg->pair_base[E] = pairs;
      if (!seg->ok && blockIdx.x == 0) latch_error(p.status, MXFP8_ERR_BAD_OFFSETS);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const int32_t ce = seg->off[e + 1] - seg->off[e];
      int rank = 0;
      for (int f = 0; f < E; ++f) {
        const int32_t cf = seg->off[f + 1] - seg->off[f];
        rank += (cf > ce) || (cf == ce && f < e);
      }
      seg->order[rank] = static_cast<int16_t>(e);
    }
  }
  if (warp == 1) tmem_alloc_2sm(tmem_slot, D::kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA copy, arrive or commit
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if constexpr (!D::kGrouped) grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer (both)
    // whole warp in the loop (warp-uniform addresses), one elected lane issues the copies
    const bool issuer = elect_one();
    const uint32_t full0 = cluster_map(&full[0], 0);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t id = first_id; ok; id += id_step) {
      const DuoTile t = duo_tile_of<BN, kMode, kSplit>(p, seg, id, crank);
      if (!t.live) break;
      const bool whole = t.width == BN;
      const uint32_t tx = whole ? D::kStageBytes : D::kHalfStageBytes;
      for (int64_t kb = 0; kb < t.nk; ++kb, ++it) {
        const uint32_t s = it % kStages, ph = (it / kStages) & 1;
        if (!warp_wait(&empty[s], ph ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
        const uint32_t bar = full0 + 8 * s;
        const int64_t kg = t.kb0 + kb;  // K stage within the whole tile
        const int32_t kx = static_cast<int32_t>(t.k_origin + kg * BK);
        if (issuer) {
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * tx);
          tma_load_2d_2sm(smem + D::kOffA + s * D::kABytes, &map_a, kx,
                          static_cast<int32_t>(t.m0), bar);
          if constexpr (kMode == kGroupRows && D::kWide) {
            // expert b_z's rows 96c.. of each 192-column half of the pair tile
            uint8_t* bs = smem + D::kOffB + s * D::kBBytes;
            tma_load_3d_2sm(bs, &map_b, kx, static_cast<int32_t>(t.n0 + 96 * crank), t.b_z, bar);
            tma_load_3d_2sm(bs + 96 * BK, &map_b, kx,
                            static_cast<int32_t>(t.n0 + 192 + 96 * crank), t.b_z, bar);
          } else if constexpr (kMode == kGroupRows) {
            tma_load_3d_2sm(smem + D::kOffB + s * D::kBBytes, &map_b, kx,
                            static_cast<int32_t>(t.n0 + crank * (BN / 2)), t.b_z, bar);
          } else if constexpr (D::kWide) {
            // rows 96c.. of each 192-column half of the pair tile; a half tile (its first
            // MMA alone) loads the first box only
            uint8_t* bs = smem + D::kOffB + s * D::kBBytes;
            tma_load_2d_2sm(bs, &map_b, kx, static_cast<int32_t>(t.n0 + 96 * crank), bar);
            if (whole)
              tma_load_2d_2sm(bs + 96 * BK, &map_b, kx,
                              static_cast<int32_t>(t.n0 + 192 + 96 * crank), bar);
          } else {
            tma_load_2d_2sm(smem + D::kOffB + s * D::kBBytes, &map_b, kx,
                            static_cast<int32_t>(t.n0 + crank * (t.width / 2)), bar);
          }
          if constexpr (kMode == kDense) {
            tma_load_3d_2sm(smem + D::kOffSfa + s * D::kSfaBytes, &map_sfa, 0,
                            static_cast<int32_t>(kg), static_cast<int32_t>(t.mt), bar);
            tma_load_3d_2sm(smem + D::kOffSfb + s * D::kSfbBytes, &map_sfb, 0,
                            static_cast<int32_t>(kg), static_cast<int32_t>(t.sfb_tile), bar);
          } else {  // scale tiles by flat index, one 512-byte tile per load
            tma_load_2d_2sm(smem + D::kOffSfa + s * D::kSfaBytes, &map_sfa, 0,
                            static_cast<int32_t>(t.sfa_idx + kb), bar);
            tma_load_2d_2sm(smem + D::kOffSfb + s * D::kSfbBytes, &map_sfb, 0,
                            static_cast<int32_t>(t.sfb_idx0 + kb), bar);
            tma_load_2d_2sm(smem + D::kOffSfb + s * D::kSfbBytes + 512, &map_sfb, 0,
                            static_cast<int32_t>(t.sfb_idx1 + kb), bar);
            if constexpr (D::kWide)
              tma_load_2d_2sm(smem + D::kOffSfb + s * D::kSfbBytes + 1024, &map_sfb, 0,
                              static_cast<int32_t>(t.sfb_idx2 + kb), bar);
          }
        }
        __syncwarp();
      }
    }
    if (!ok && issuer) {
      *abort_flag = 1;
      latch_error(p.status, MXFP8_ERR_TIMEOUT);
    }
    // the copies still in flight are waited for on the way out, by the leader, whose full
    // barriers count both CTAs' bytes; both CTAs learn what each producer issued
    if (issuer)
      for (uint32_t r = 0; r < 2; ++r)
        st_cluster_u32(cluster_map(const_cast<uint32_t*>(&rec[crank]), r), it);
    // Producer tail: the leader's release (a multicast commit) of the last stage uses must
    // have arrived on this CTA's empty barriers before it exits; those arrivals can land
    // after the epilogue has seen the last accumulator. Waiting here overlaps the epilogue's
    // last tile; after an abort the drain below does it instead.
    bool tail_ok = ok;
    for (uint32_t i = it > kStages ? it - kStages : 0; tail_ok && i < it; ++i)
      tail_ok = warp_wait(&empty[i % kStages], (i / kStages) & 1, abort_flag, p.wait_ns);
    if (issuer) rec[4] = tail_ok ? 1u : 0u;
    __syncwarp();
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------- MMA issuer (leader)
    // whole warp in the loop (warp-uniform descriptors), one elected lane issues
    const bool issuer = elect_one();
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    const uint64_t a_desc0 = smem_desc(smem_u32(smem + D::kOffA), 16, 1024, 2);
    const uint64_t b_desc0 = smem_desc(smem_u32(smem + D::kOffB), 16, 1024, 2);
    const uint64_t sfa_desc0 = smem_desc(smem_u32(smem + D::kOffSfa), 0, 128, 0);
    const uint64_t sfb_desc0 = smem_desc(smem_u32(smem + D::kOffSfb), 0, 128, 0);
    constexpr int kN = D::kMmaN;
    constexpr uint32_t kId0 = mxf8_idesc(2 * BM, kN, 0, 0), kId1 = mxf8_idesc(2 * BM, kN, 1, 1);
    constexpr uint32_t kId2 = mxf8_idesc(2 * BM, kN, 2, 2), kId3 = mxf8_idesc(2 * BM, kN, 3, 3);
    // half tiles of the 256-wide kernel: N = 128, the same B scale bytes (their columns
    // start at a 128-row tile); a 384-wide kernel's half tile is its first MMA alone
    constexpr uint32_t kHalfN = D::kWide ? 0u : (mxf8_idesc(2 * BM, BN / 2, 0, 0) ^ kId0);
    for (int64_t id = first_id; ok; id += id_step) {
      const DuoTile t = duo_tile_of<BN, kMode, kSplit>(p, seg, id, crank);
      if (!t.live) break;
      if (t.nk == 0) continue;  // an empty expert's dW tile: the epilogue writes zeros
      const uint32_t buf = acc_it % D::kAcc, aph = (acc_it / D::kAcc) & 1;
      if (!warp_wait(&acc_empty[buf], aph ^ 1, abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_t = tmem + buf * BN;
      const uint32_t shift = static_cast<uint32_t>(t.sfb_shift);
      const uint32_t nx = t.width == BN ? 0u : kHalfN;  // flips the N field to BN / 2
      const bool second = D::kWide && t.width == BN;     // the columns [192, 384) too
      for (int64_t kb = 0; kb < t.nk; ++kb, ++it) {
        const uint32_t s = it % kStages, ph = (it / kStages) & 1;
        if (!warp_wait(&full[s], ph, abort_flag, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sfa_t = tmem + D::kSfaCol + 4 * s;
        const uint32_t sfb_slot = tmem + D::kSfbCol + D::kSfbSlot * s;
        const uint32_t sfb_t = sfb_slot + shift;  // B rows 0-31 of the tile
        const uint64_t sbd = sfb_desc0 + s * (D::kSfbBytes / 16);
        const uint64_t ad = a_desc0 + s * (D::kABytes / 16);
        const uint64_t bd = b_desc0 + s * (D::kBBytes / 16);
        const uint32_t acc0 = kb > 0 ? 1u : 0u;
        if (issuer) {
          tmem_cp_32x128b_x4_2sm(sfa_t, sfa_desc0 + s * (D::kSfaBytes / 16));
          tmem_cp_32x128b_x4_2sm(sfb_slot, sbd);
          tmem_cp_32x128b_x4_2sm(sfb_slot + 4, sbd + 512 / 16);
          if constexpr (D::kWide) tmem_cp_32x128b_x4_2sm(sfb_slot + 8, sbd + 1024 / 16);
          // 384-wide: the second MMA's B rows start 96 rows into the stage, its scales 192
          // rows into the slot (column 6: 64 rows into the second scale tile)
          const uint64_t bd2 = bd + (96 * BK) / 16;
          const uint32_t d_t2 = d_t + 192, sfb_t2 = sfb_slot + 6;
          if (kb != t.nk - 1 || t.last_blocks == 4) {
            mma_mxf8_2sm(d_t, ad, bd, kId0 ^ nx, sfa_t, sfb_t, acc0);
            mma_mxf8_2sm(d_t, ad + 2, bd + 2, kId1 ^ nx, sfa_t, sfb_t, 1u);
            mma_mxf8_2sm(d_t, ad + 4, bd + 4, kId2 ^ nx, sfa_t, sfb_t, 1u);
            mma_mxf8_2sm(d_t, ad + 6, bd + 6, kId3 ^ nx, sfa_t, sfb_t, 1u);
            if (second) {
              mma_mxf8_2sm(d_t2, ad, bd2, kId0, sfa_t, sfb_t2, acc0);
              mma_mxf8_2sm(d_t2, ad + 2, bd2 + 2, kId1, sfa_t, sfb_t2, 1u);
              mma_mxf8_2sm(d_t2, ad + 4, bd2 + 4, kId2, sfa_t, sfb_t2, 1u);
              mma_mxf8_2sm(d_t2, ad + 6, bd2 + 6, kId3, sfa_t, sfb_t2, 1u);
            }
          } else {
            for (int k = 0; k < t.last_blocks; ++k)
              mma_mxf8_2sm(d_t, ad + 2 * k, bd + 2 * k, mxf8_idesc(2 * BM, kN, k, k) ^ nx,
                           sfa_t, sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
            if (second)
              for (int k = 0; k < t.last_blocks; ++k)
                mma_mxf8_2sm(d_t2, ad + 2 * k, bd2 + 2 * k, mxf8_idesc(2 * BM, kN, k, k), sfa_t,
                             sfb_t2, (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit_2sm_mc(&empty[s], 0x3);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (issuer) mma_commit_2sm_mc(&acc_full[buf], 0x3);
      __syncwarp();
      ++acc_it;
    }
    if (!ok && issuer) {
      *abort_flag = 1;
      latch_error(p.status, MXFP8_ERR_TIMEOUT);
    }
    // the pair's tensor-core work must be finished before either CTA frees its TMEM
    if (issuer) {
      for (uint32_t r = 0; r < 2; ++r) {
        st_cluster_u32(cluster_map(const_cast<uint32_t*>(&rec[2]), r), it);
        st_cluster_u32(cluster_map(const_cast<uint32_t*>(&rec[3]), r), acc_it);
      }
      mma_commit_2sm_mc(mma_done, 0x1);
      mbar_wait_timed(mma_done, 0, p.drain_ns);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ------------------------------------------------------------- epilogue (both)
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the BN columns
    constexpr int kChunks = BN / 64;   // 32-column chunks per warp
    const uint32_t acc_empty0 = cluster_map(&acc_empty[0], 0);
    uint8_t* box = smem + D::kOffOut + (warp - 2) * D::kStageBoxBytes;
    uint32_t acc_it = 0;
    bool ok = true;
    for (int64_t id = first_id; ok; id += id_step) {
      const DuoTile t = duo_tile_of<BN, kMode, kSplit>(p, seg, id, crank);
      if (!t.live) break;
      if constexpr (D::kWide) {
        // 384-wide (BF16 out): 6 chunks of 32 columns per warp, converted to BF16 pairs as
        // they leave TMEM in 3 rounds of 2 chunks, so that the accumulator is handed back
        // before any store; then 32-byte boxes (16 columns) with the 32-byte swizzle.
        // One 32-row x 16-column box of BF16 pairs (lo: columns 0-7, hi: 8-15) through the
        // warp's staging box, 16-byte chunks swapped on alternate row groups (32-byte swizzle).
        auto store_box = [&](uint4 lo, uint4 hi, int col) {
          const int sw = (lane >> 2) & 1;
          if (lane == 0) bulk_wait_read_all();  // the box is free again
          __syncwarp();
          *reinterpret_cast<uint4*>(box + lane * 32 + 16 * sw) = lo;
          *reinterpret_cast<uint4*>(box + lane * 32 + 16 * (sw ^ 1)) = hi;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&map_c, box, static_cast<int32_t>(t.n0 + col),
                         static_cast<int32_t>(t.m0 + 32 * q));
            bulk_commit_group();
          }
        };
        if constexpr (kSplit) if (t.piece >= 0) {
          // A split-K piece (the host gives each at least one stage). Pieces other than the
          // last write their FP32 accumulator to the workspace and count themselves in on
          // the warp's arrival counter (a release); the last piece waits until all have
          // arrived, sets the counter back to zero for the next launch (or graph replay),
          // and adds the partials before converting, round by round, storing each round
          // at once (its tile is the CTA's last: holding the accumulator a little longer
          // delays nothing). Workspace layout, in 32-byte units: [tile slot][piece][CTA
          // rank][epilogue warp][round][column group of 8][lane], so that a warp's 32-byte
          // stores cover 1 KB contiguous and each lane reads back what the same lane of the
          // same warp wrote.
          constexpr int S = kSplitK;
          const bool writer = t.piece < S - 1;
          const int ew = warp - 2;
          auto ws_at = [&](int piece, int r) {  // this lane's first 32-byte unit of round r
            return reinterpret_cast<uint8_t*>(p.ws) +
                   (((((static_cast<size_t>(t.slot) * (S - 1) + piece) * 2 + crank) * kEpiWarps +
                      ew) * 3 + r) * (8 * 32) + lane) * 32;
          };
          uint32_t* const count = p.ws_flags + (static_cast<size_t>(t.slot) * 2 + crank) * kEpiWarps + ew;
          int got = 0;
          if (lane == 0) got = mbar_wait_bounded(&acc_full[0], acc_it & 1, abort_flag, p.wait_ns);
          if (!writer && lane == 0 && got)
            got = flag_wait_bounded(count, S - 1, abort_flag, p.wait_ns);
          got = __shfl_sync(0xFFFFFFFFu, got, 0);
          if (!got) { ok = false; break; }
          if (!writer) {
            (void)ld_acquire_gpu(count);  // every lane
            __syncwarp();
            if (lane == 0) *count = 0;    // every writer of this launch has arrived
          }
          tc_fence_after();
          __syncwarp();
          const uint32_t base = tmem + (static_cast<uint32_t>(32 * q) << 16) + half * 192;
#pragma unroll 1
          for (int r = 0; r < 3; ++r) {
            uint32_t v[2][32];
            tmem_ld_32x32b_x32(base + 64 * r, v[0]);
            tmem_ld_32x32b_x32(base + 64 * r + 32, v[1]);
            tmem_ld_wait();
            if (writer) {
              uint8_t* w = ws_at(t.piece, r);
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                const int u = g >> 2, c = 8 * (g & 3);
                st_global_cg_v8(w + g * (32 * 32), v[u][c], v[u][c + 1], v[u][c + 2], v[u][c + 3],
                                v[u][c + 4], v[u][c + 5], v[u][c + 6], v[u][c + 7]);
              }
              continue;
            }
#pragma unroll
            for (int pp = 0; pp < S - 1; ++pp) {
              const uint8_t* w = ws_at(pp, r);
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                uint32_t x[8];
                ld_global_cg_v8(w + g * (32 * 32), x);
                const int u = g >> 2, c = 8 * (g & 3);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  v[u][c + j] = __float_as_uint(__uint_as_float(v[u][c + j]) + __uint_as_float(x[j]));
              }
            }
            if (32 * q < t.rows_valid) {
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                uint32_t bb[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  bb[i] = cvt_bf16x2(__uint_as_float(v[u][2 * i + 1]), __uint_as_float(v[u][2 * i]));
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                  const int col = 32 * (half * 6 + 2 * r + u) + 16 * g;
                  if (col < t.cols_valid)
                    store_box(make_uint4(bb[8 * g], bb[8 * g + 1], bb[8 * g + 2], bb[8 * g + 3]),
                              make_uint4(bb[8 * g + 4], bb[8 * g + 5], bb[8 * g + 6], bb[8 * g + 7]),
                              col);
                }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty0);
          ++acc_it;
          if (writer) {  // the partial is out: release it to the last piece
            __threadfence();
            __syncwarp();
            if (lane == 0) red_release_add_gpu(count, 1u);
          }
          continue;
        }
        uint32_t b[6][16];
        if (t.nk > 0) {
          const uint32_t aph = acc_it & 1;
          int got = 0;
          if (lane == 0) got = mbar_wait_bounded(&acc_full[0], aph, abort_flag, p.wait_ns);
          got = __shfl_sync(0xFFFFFFFFu, got, 0);
          if (!got) { ok = false; break; }
          tc_fence_after();
          __syncwarp();
          const uint32_t base = tmem + (static_cast<uint32_t>(32 * q) << 16) + half * 192;
#pragma unroll
          for (int r = 0; r < 3; ++r) {
            uint32_t v[2][32];
            tmem_ld_32x32b_x32(base + 64 * r, v[0]);
            tmem_ld_32x32b_x32(base + 64 * r + 32, v[1]);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int i = 0; i < 16; ++i)
                b[2 * r + u][i] = cvt_bf16x2(__uint_as_float(v[u][2 * i + 1]),
                                             __uint_as_float(v[u][2 * i]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty0);
          ++acc_it;
        } else {
#pragma unroll
          for (int c = 0; c < 6; ++c)
#pragma unroll
            for (int i = 0; i < 16; ++i) b[c][i] = 0;
        }
        if (32 * q < t.rows_valid) {
          const int sw = (lane >> 2) & 1;
#pragma unroll
          for (int c6 = 0; c6 < 6; ++c6) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const int col = 32 * (half * 6 + c6) + 16 * g;  // first column of this box
              if (col >= t.cols_valid) continue;
              if (lane == 0) bulk_wait_read_all();  // the box is free again
              __syncwarp();
              *reinterpret_cast<uint4*>(box + lane * 32 + 16 * sw) =
                  make_uint4(b[c6][8 * g], b[c6][8 * g + 1], b[c6][8 * g + 2], b[c6][8 * g + 3]);
              *reinterpret_cast<uint4*>(box + lane * 32 + 16 * (sw ^ 1)) =
                  make_uint4(b[c6][8 * g + 4], b[c6][8 * g + 5], b[c6][8 * g + 6], b[c6][8 * g + 7]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&map_c, box, static_cast<int32_t>(t.n0 + col),
                             static_cast<int32_t>(t.m0 + 32 * q));
                bulk_commit_group();
              }
            }
          }
        }
        continue;
      }
      // The whole slice goes to registers and TMEM is handed back before any store.
      uint32_t v[kChunks][32];
      if (t.nk > 0) {
        const uint32_t buf = acc_it % D::kAcc, aph = (acc_it / D::kAcc) & 1;
        int got = 0;
        if (lane == 0) got = mbar_wait_bounded(&acc_full[buf], aph, abort_flag, p.wait_ns);
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) { ok = false; break; }
        tc_fence_after();
        __syncwarp();
        const uint32_t base =
            tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * BN + half * kChunks * 32;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tmem_ld_32x32b_x32(base + 32 * c, v[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty0 + 8 * buf);
        ++acc_it;
      } else {  // an empty expert: its dW tile is zero
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[c][i] = 0;
      }
      // Stores leave through shared memory: each 64-byte column group of the warp's 32 rows
      // is written into the warp's staging box (16-byte chunks XOR-swizzled as the tensor
      // map's 64-byte swizzle expects, so the 32 lanes hit distinct banks) and sent with one
      // TMA store, which clips rows and columns past the matrix. One thread-row per lane
      // would otherwise touch 32 cache lines per store instruction.
      if (32 * q < t.rows_valid) {
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const int c = half * kChunks + u;
          if (32 * c >= t.cols_valid) continue;
#pragma unroll
          for (int g = 0; g < (p.out_fp32 ? 2 : 1); ++g) {
            uint4 w[4];
            if (p.out_fp32) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                w[j] = make_uint4(v[u][16 * g + 4 * j], v[u][16 * g + 4 * j + 1],
                                  v[u][16 * g + 4 * j + 2], v[u][16 * g + 4 * j + 3]);
            } else {
              uint32_t b[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                b[i] = cvt_bf16x2(__uint_as_float(v[u][2 * i + 1]), __uint_as_float(v[u][2 * i]));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                w[j] = make_uint4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
            }
            const int col = 32 * c + 16 * g;  // first column of this group
            if (p.out_fp32 && col >= t.cols_valid) continue;
            if (lane == 0) bulk_wait_read_all();  // the box is free again
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(box + lane * 64 + 16 * (j ^ ((lane >> 1) & 3))) = w[j];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if constexpr (kMode == kDense)
                tma_store_2d(&map_c, box, static_cast<int32_t>(t.n0 + col),
                             static_cast<int32_t>(t.m0 + 32 * q));
              else
                tma_store_3d(&map_c, box, static_cast<int32_t>(t.n0 + col),
                             static_cast<int32_t>(t.m0 + 32 * q), t.c_z);
              bulk_commit_group();
            }
          }
        }
      }
    }
    // Before the CTA exits its stores must have finished reading its shared memory; the
    // kernel's completion makes their global writes visible to later work.
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    if (!ok && lane == 0) {
      *abort_flag = 1;
      latch_error(p.status, MXFP8_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs have stopped issuing; the drain records are in place
  // Drain: whatever stopped the loops, no copy, MMA or commit of the pair may still be
  // landing in either CTA when it exits. The leader completes the stage uses that only one
  // CTA issued - the missing half of the bytes is completed by hand (mbarrier complete_tx),
  // a missing arm by an arrive that expects the peer's half alone - and waits for each of
  // them to land, so both CTAs' copies are in. Each CTA then waits for the last arrival of
  // the MMA issuer's commits on its own empty and accumulator barriers. The waits have
  // their own limit, never shorter than the pipeline's.
  // Without an abort every issued stage use was consumed, the producer's tail has seen the
  // last releases and the epilogue every accumulator commit: nothing is left to wait for,
  // and the second cluster barrier is skipped (both CTAs read the same issue counts, so
  // they take the same branch).
  const uint32_t i0 = rec[0], i1 = rec[1], consumed = rec[2], commits = rec[3];
  const uint32_t issued = i0 > i1 ? i0 : i1;
  if (threadIdx.x == 0 && !(rec[4] && !*abort_flag && issued == consumed)) {
    if (leader) {
      for (uint32_t i = consumed; i < issued; ++i) {
        uint64_t* b = &full[i % kStages];
        const bool only0 = i < i0 && i >= i1, only1 = i >= i0 && i < i1;
        if (!only0 && !only1) continue;
        const uint32_t bytes =
            duo_use_bytes<BN, kMode, kSplit>(p, seg, first_id, id_step, crank, i);
        if (only0) mbar_complete_tx(b, bytes);
        else mbar_arrive_expect_tx(b, bytes);
      }
      drain_stages<kStages, D::kAcc>(full, empty, acc_full, issued, consumed, commits,
                                     p.drain_ns);
    } else {
      drain_stages<kStages, D::kAcc>(full, empty, acc_full, 0, consumed, commits, p.drain_ns);
    }
  }
  __syncthreads();
  if (issued > consumed) cluster_sync();  // the leader's drain covered the peer's copies too
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_2sm(tmem, D::kTmemCols);
  }
}

// ------------------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Row-major u8 matrix [outer][inner] (optionally [depth][outer][inner]) viewed through a
// box of box_inner bytes x box_outer rows with the 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int rank, uint64_t inner, uint64_t outer,
              uint64_t depth, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, outer, depth};
  cuuint64_t strides[2] = {inner, inner * outer};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Pipeline wait limit: mxfp8_set_wait_limit_ns, else MXFP8_WAIT_LIMIT_MS, else 4 s.
std::atomic<uint64_t> g_wait_override_ns{0};

uint64_t wait_limit_ns() {
  static const uint64_t dflt = [] {
    const char* e = getenv("MXFP8_WAIT_LIMIT_MS");
    long ms = e ? atol(e) : 0;
    if (ms <= 0) ms = 4000;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  const uint64_t o = g_wait_override_ns.load(std::memory_order_relaxed);
  return o ? o : dflt;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("MXFP8_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

}  // namespace

int pdl_attr(cudaLaunchAttribute* attr) {
  if (!pdl_enabled()) return 0;
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  return 1;
}

namespace {

// The drain waits for work already in flight on the way out of a kernel: at least 2 s, and
// never shorter than the pipeline limit, so that a short pipeline limit cannot cut them.
constexpr uint64_t kMinDrainNs = 2000000000ull;

uint64_t drain_limit_ns(uint64_t wait_ns) { return wait_ns > kMinDrainNs ? wait_ns : kMinDrainNs; }

template <int BN, int kMode>
int launch(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc, const Params& p,
           int64_t grid, cudaStream_t stream) {
  using C = Cfg<BN>;
  auto k = mxfp8_gemm_kernel<BN, kMode>;
  static std::atomic<bool> attr_set[64] = {};  // per device; setting it twice is harmless
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
      return MXFP8_ERR_CUDA;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  if (grid <= 0) return MXFP8_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  return cudaLaunchKernelEx(&cfg, k, ma, mb, mc, p) == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

// Raster band width, in M tiles. Tiles of a band are visited M tile first, so that while
// the band sweeps across N, its A row tiles stay in L2 and each B tile is fetched from
// DRAM once per band. When A is the smaller operand (M <= N) the band is as tall as
// kBandBytes of A allows, up to all of M, so that B is streamed from DRAM about once.
// Otherwise B is the smaller operand: narrow bands of 8 tiles keep all of B in L2 while
// A streams through.
constexpr int64_t kBandBytes = int64_t(48) << 20;

int band_tiles(int64_t M, int64_t N, int64_t K, int num_m_tiles) {
  int64_t gm = 8;
  if (M <= N) {
    const int64_t fit = kBandBytes / (static_cast<int64_t>(BM) * K);
    gm = fit > gm ? fit : gm;
  }
  return static_cast<int>(gm < num_m_tiles ? gm : num_m_tiles);
}

// The swizzled scales of an operand as a 3-D tensor [row tiles][K tiles][512 bytes], read
// as 16-bit elements so that one 512-byte scale tile is a single box row.
bool make_sf_map(CUtensorMap* map, const void* base, int64_t row_tiles, int64_t k_tiles,
                 uint32_t tiles_per_box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {256, static_cast<cuuint64_t>(k_tiles), static_cast<cuuint64_t>(row_tiles)};
  cuuint64_t strides[2] = {512, static_cast<cuuint64_t>(k_tiles) * 512};
  cuuint32_t box[3] = {256, 1, tiles_per_box};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The output C [Z][rows][N] (BF16 or FP32; rank 2 when Z == 1 and rank == 2) for TMA
// stores of 32-row boxes of `row_bytes` (64 or 32) with the swizzle of the same width.
bool make_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t N, int64_t Z, bool fp32,
                  int rank, uint32_t row_bytes = 64) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint32_t elem = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(Z)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * elem,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(rows) * elem};
  cuuint32_t box[3] = {row_bytes / elem, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
            static_cast<cuuint32_t>(rank), base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaLaunchConfig_t cluster2_config(int64_t grid, int smem, cudaStream_t stream,
                                   cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// How many clusters of the 2SM kernel fit on the device at once (cached per device).
template <int BN, int kMode = kDense>
int64_t max_duo_clusters() {
  static std::atomic<int64_t> cached[64] = {};  // per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int64_t c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  auto k = mxfp8_gemm_2sm_kernel<BN, kMode>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Duo<BN, kMode>::kSmemBytes) != cudaSuccess)
    return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster2_config(2 * 256, Duo<BN, kMode>::kSmemBytes, nullptr, attr);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, k, &cfg) != cudaSuccess || clusters <= 0)
    clusters = num_sms() / 2;
  if (dev >= 0 && dev < 64) cached[dev].store(clusters, std::memory_order_relaxed);
  return clusters;
}

// Dense GEMMs with N > 128 and at least two M tiles run on the 2SM kernel;
// MXFP8_GEMM_2SM=0 selects the one-SM kernel instead.
bool duo_enabled() {
  static const bool on = [] {
    const char* e = getenv("MXFP8_GEMM_2SM");
    return !(e && e[0] == '0');
  }();
  return on;
}

// 384-wide tiles for dense BF16-output GEMMs; MXFP8_GEMM_WIDE=0 turns them off.
bool wide_tiles_enabled() {
  static const bool on = [] {
    const char* e = getenv("MXFP8_GEMM_WIDE");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Half-width tiles for the last wave of the 256- and 384-wide 2SM kernel;
// MXFP8_GEMM_HALF_TAIL=0 turns them off.
bool half_tail_enabled() {
  static const bool on = [] {
    const char* e = getenv("MXFP8_GEMM_HALF_TAIL");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Tile width of the 2SM kernel for one problem: 192, 256 or 384 (BF16 output only), the
// one with the least estimated time. A tile's time per K stage relative to a 256-wide tile,
// as measured on GB300 (narrow tiles pay the per-stage scale copies and fills over fewer
// FLOPs; the 384-wide tile, two MMAs sharing A, is slightly cheaper per FLOP): 192 -> 0.78,
// 256 -> 1, 384 -> 1.46; a last wave of half tiles costs 0.93 (256) or 0.78 (384, two
// 192-wide halves). MXFP8_GEMM_BN=192, 256 or 384 forces a width.
int duo_width(int64_t M, int64_t N, bool fp32) {
  static const int forced = [] {
    const char* e = getenv("MXFP8_GEMM_BN");
    const int w = e ? atoi(e) : 0;
    return (w == 256 || w == 192 || w == 384) ? w : 0;
  }();
  if (forced && !(forced == 384 && fp32)) return forced;
  const int64_t clusters = num_sms() / 2;
  auto cost = [&](int bn) {
    const double full = bn == 192 ? 0.78 : (bn == 256 ? 1.0 : 1.46);
    const double halfc = bn == 256 ? 0.93 : 0.78;
    const int64_t tiles = ((M + 255) / 256) * ((N + bn - 1) / bn);
    const int64_t waves = tiles / clusters, tail = tiles % clusters;
    double t = static_cast<double>(waves) * full;
    if (tail > 0)
      t += (bn != 192 && half_tail_enabled() && 2 * tail <= clusters) ? halfc : full;
    return t;
  };
  int best = 256;
  double best_t = cost(256);
  const int others[2] = {192, 384};
  for (int bn : others) {
    if (bn == 384 && (fp32 || !wide_tiles_enabled())) continue;
    const double t = cost(bn);
    if (t < best_t) best = bn, best_t = t;
  }
  return best;
}

// Split-K last waves: a 384-wide kernel's partial last wave of `tail` pair tiles runs as
// kSplitK K pieces per tile (instead of two half tiles) when the pieces fit in one wave
// and every piece gets at least kSplitKMinStages K stages. The workspace holds the FP32
// partials of kSplitK - 1 pieces per tile (the last piece adds them) and one arrival
// counter per tile, CTA rank and epilogue warp. Measured on 4096 x 4096 x K (GB300): the
// pieces run at about 600 ns per stage against 307 for a half tile, and the reduction
// costs about 10 us, so split-K wins only on deep reductions. At K = 24576 it takes 245 to 235 us;
// at K = 12288 it breaks even; at K <= 8192 it loses.
constexpr int kSplitKMinStages = 40;  // per piece; MXFP8_GEMM_SPLITK_MIN_STAGES overrides
constexpr size_t kSplitKPartialBytes = size_t(2) * BM * 384 * 4;  // FP32, one pair tile
constexpr size_t kSplitKFlagBytes = size_t(2) * kEpiWarps * 4;  // one tile's counters

struct SplitPlan {
  int64_t tail = 0;      // split tiles (0: no split-K)
  size_t bytes = 0;      // workspace bytes it needs
};

SplitPlan split_plan(int64_t pair_tiles, int64_t fit, int64_t n_kt) {
  SplitPlan s;
  static const bool on = [] {
    const char* e = getenv("MXFP8_GEMM_SPLITK");
    return !(e && e[0] == '0');
  }();
  static const int64_t min_stages = [] {
    const char* e = getenv("MXFP8_GEMM_SPLITK_MIN_STAGES");
    const long v = e ? atol(e) : 0;
    return static_cast<int64_t>(v >= 1 ? v : kSplitKMinStages);
  }();
  const int64_t tail = pair_tiles % fit;
  if (!on || tail == 0 || kSplitK * tail > fit || n_kt < kSplitK * min_stages) return s;
  s.tail = tail;
  s.bytes = static_cast<size_t>(tail) * ((kSplitK - 1) * kSplitKPartialBytes + kSplitKFlagBytes);
  return s;
}

// Dense GEMM on CTA pairs with 256 x BN tiles (tcgen05 cta_group::2).
template <int BN>
int launch_duo(const GemmArgs& a, Params p, cudaStream_t stream) {
  using D = Duo<BN>;
  const int64_t n_kt = (a.K + BK - 1) / BK;
  CUtensorMap ma, mb, msa, msb, mc;
  if (!make_map(&ma, a.A, 2, a.K, a.M, 1, BK, BM)) return MXFP8_ERR_CUDA;
  if (D::kWide && a.out_dtype == MXFP8_OUT_FP32) return MXFP8_ERR_INVALID_ARG;
  if (!make_map(&mb, a.B, 2, a.K, a.N, 1, BK, D::kBoxRows)) return MXFP8_ERR_CUDA;
  if (!make_out_map(&mc, a.C, a.M, a.N, 1, a.out_dtype == MXFP8_OUT_FP32, 2, D::kBoxRowBytes))
    return MXFP8_ERR_CUDA;
  if (!make_sf_map(&msa, a.sA, (a.M + 127) / 128, n_kt, 1)) return MXFP8_ERR_CUDA;
  if (!make_sf_map(&msb, a.sB, (a.N + 127) / 128, n_kt, D::kSfbTiles)) return MXFP8_ERR_CUDA;
  p.num_n_tiles = static_cast<int>((a.N + BN - 1) / BN);
  p.num_tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
  p.band = (band_tiles(a.M, a.N, a.K, p.num_m_tiles) + 1) / 2;
  const int64_t pair_tiles = static_cast<int64_t>((p.num_m_tiles + 1) / 2) * p.num_n_tiles;
  if (2 * pair_tiles > INT32_MAX) return MXFP8_ERR_INVALID_ARG;  // 32-bit item arithmetic
  const int64_t fit = max_duo_clusters<BN>();
  if (fit <= 0) return MXFP8_ERR_CUDA;
  // The tiles of the last, partial wave run as split-K pieces (384-wide, deep K, with a
  // large enough workspace), else as half-width tiles when their halves still fit in one
  // wave of clusters (256- and 384-wide tiles).
  int64_t items = pair_tiles;
  const int64_t tail = pair_tiles % fit;
  const SplitPlan sp = BN == 384 ? split_plan(pair_tiles, fit, n_kt) : SplitPlan{};
  if (sp.tail > 0 && a.workspace && a.workspace_bytes >= sp.bytes &&
      (reinterpret_cast<uintptr_t>(a.workspace) & 31) == 0) {
    p.split_from = pair_tiles - tail;
    p.ws = static_cast<uint4*>(a.workspace);
    p.ws_flags = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.workspace) +
                                             static_cast<size_t>(tail) * (kSplitK - 1) *
                                                 kSplitKPartialBytes);
    items = pair_tiles + (kSplitK - 1) * tail;
  } else if (BN != 192 && half_tail_enabled() && tail > 0 && 2 * tail <= fit) {
    p.split_from = pair_tiles - tail;
    items = pair_tiles + tail;
  }
  const int64_t clusters = items < fit ? items : fit;
  if (clusters <= 0) return MXFP8_OK;
  auto k = mxfp8_gemm_2sm_kernel<BN, kDense>;
  if constexpr (BN == 384) {
    if (p.ws) {
      k = mxfp8_gemm_2sm_kernel<BN, kDense, true>;
      static std::atomic<bool> attr_set[64] = {};  // per device; setting it twice is harmless
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess) return MXFP8_ERR_CUDA;
      if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 D::kSmemBytes) != cudaSuccess)
          return MXFP8_ERR_CUDA;
        if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
      }
    }
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster2_config(2 * clusters, D::kSmemBytes, stream, attr);
  cfg.numAttrs += pdl_attr(&attr[1]);
  return cudaLaunchKernelEx(&cfg, k, ma, mb, msa, msb, mc, p) == cudaSuccess ? MXFP8_OK
                                                                              : MXFP8_ERR_CUDA;
}

// The scale tiles of an operand as a flat array of 512-byte tiles (16-bit elements), for
// grouped layouts whose K-tile count differs from expert to expert.
bool make_sf_flat_map(CUtensorMap* map, const void* base, int64_t tiles) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(tiles)};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {256, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Grouped GEMM on CTA pairs (kGroupRows: fprop/dgrad, kGroupWgrad). `p` has M, N, K, E,
// offsets and total_rows set as the one-SM grouped launcher sets them.
template <int BN, int kMode>
int launch_duo_grouped(const GemmArgs& a, Params p, cudaStream_t stream) {
  using D = Duo<BN, kMode>;
  const int64_t T = p.total_rows, E = p.E;
  const int64_t seg_tiles = (T + 127) / 128 + E;  // bound on sum of ceil(count / 128)
  const bool fp32 = p.out_fp32 != 0;
  CUtensorMap ma, mb, msa, msb, mc;
  int64_t pair_tiles = 0;
  p.num_n_tiles = static_cast<int>((p.N + BN - 1) / BN);
  if (kMode == kGroupWgrad) {
    // A = dY^T [M][T], B = X^T [N][T], both blocked along the tokens; C[e] = [M][N]
    if (!make_map(&ma, a.A, 2, T, p.M, 1, BK, BM)) return MXFP8_ERR_CUDA;
    if (!make_map(&mb, a.B, 2, T, p.N, 1, BK, D::kBoxRows)) return MXFP8_ERR_CUDA;
    if (!make_sf_flat_map(&msa, a.sA, ((p.M + 127) / 128) * seg_tiles)) return MXFP8_ERR_CUDA;
    if (!make_sf_flat_map(&msb, a.sB, ((p.N + 127) / 128) * seg_tiles)) return MXFP8_ERR_CUDA;
    if (!make_out_map(&mc, a.C, p.M, p.N, E, fp32, 3)) return MXFP8_ERR_CUDA;
    pair_tiles = (((p.M + 127) / 128 + 1) / 2) * p.num_n_tiles * E;
  } else {
    // A = X [T][K] segmented by rows, B = W [E][N][K], C = [T][N]
    const int64_t n_kt = (p.K + BK - 1) / BK;
    if (!make_map(&ma, a.A, 2, p.K, T, 1, BK, BM)) return MXFP8_ERR_CUDA;
    if (!make_map(&mb, a.B, 3, p.K, p.N, E, BK, D::kBoxRows)) return MXFP8_ERR_CUDA;
    if (!make_sf_flat_map(&msa, a.sA, seg_tiles * n_kt)) return MXFP8_ERR_CUDA;
    if (!make_sf_flat_map(&msb, a.sB, E * ((p.N + 127) / 128) * n_kt)) return MXFP8_ERR_CUDA;
    // 384-wide tiles store 32-byte boxes through a 2-D map (the wide epilogue's path)
    if (D::kWide ? !make_out_map(&mc, a.C, T, p.N, 1, fp32, 2, D::kBoxRowBytes)
                 : !make_out_map(&mc, a.C, T, p.N, 1, fp32, 3))
      return MXFP8_ERR_CUDA;
    pair_tiles = ((T + 127) / 128 / 2 + E) * p.num_n_tiles;  // bound on pair tiles
  }
  if (pair_tiles > INT32_MAX) return MXFP8_ERR_INVALID_ARG;  // 32-bit item arithmetic
  const int64_t fit = max_duo_clusters<BN, kMode>();
  if (fit <= 0) return MXFP8_ERR_CUDA;
  const int64_t clusters = pair_tiles < fit ? pair_tiles : fit;
  if (clusters <= 0) return MXFP8_OK;
  auto k = mxfp8_gemm_2sm_kernel<BN, kMode>;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster2_config(2 * clusters, D::kSmemBytes, stream, attr);
  cfg.numAttrs += pdl_attr(&attr[1]);
  return cudaLaunchKernelEx(&cfg, k, ma, mb, msa, msb, mc, p) == cudaSuccess ? MXFP8_OK
                                                                              : MXFP8_ERR_CUDA;
}

// Tile width for the grouped 2SM GEMMs: 256 (measured faster than 192 for both modes on
// the Qwen3-30B-A3B expert layer, wgrad included), or 384 for fprop / dgrad with BF16 output
// when N is a multiple of 384 of at least 4 tiles. On that layer 384 took gate_up fprop
// (N = 1536) from 174.5 to 170.2 us, and down dgrad (N = 768, 2 tiles) from 96.7 to 97.5.
// MXFP8_GEMM_BN forces a width; a forced 384 applies to any multiple of 384.
int duo_grouped_width(int mode, int64_t N, bool fp32) {
  const char* e = getenv("MXFP8_GEMM_BN");
  const int w = e ? atoi(e) : 0;
  const bool wide_ok = mode == kGroupRows && !fp32 && N % 384 == 0 && wide_tiles_enabled();
  if (w == 256 || w == 192) return w;
  if (w == 384) return wide_ok ? 384 : 256;
  return wide_ok && N >= 4 * 384 ? 384 : 256;
}

}  // namespace

void set_wait_limit_ns(uint64_t ns) { g_wait_override_ns.store(ns, std::memory_order_relaxed); }

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int out_dtype) {
  const bool fp32 = out_dtype == MXFP8_OUT_FP32;
  const int64_t num_m_tiles = (M + BM - 1) / BM;
  if (N <= 128 || num_m_tiles < 2 || !duo_enabled() || duo_width(M, N, fp32) != 384) return 0;
  const int64_t fit = max_duo_clusters<384>();
  if (fit <= 0) return 0;
  const int64_t pair_tiles = ((num_m_tiles + 1) / 2) * ((N + 383) / 384);
  return split_plan(pair_tiles, fit, (K + BK - 1) / BK).bytes;
}

int launch_gemm(const GemmArgs& a, cudaStream_t stream) {
  Params p{};
  p.sA = static_cast<const uint8_t*>(a.sA);
  p.sB = static_cast<const uint8_t*>(a.sB);
  p.C = a.C;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.out_fp32 = a.out_dtype == MXFP8_OUT_FP32;
  p.status = a.status;
  p.wait_ns = wait_limit_ns();
  p.drain_ns = drain_limit_ns(p.wait_ns);
  const bool wide = a.N > 128;
  const int bn = wide ? 256 : 128;
  p.num_m_tiles = static_cast<int>((a.M + BM - 1) / BM);
  p.num_n_tiles = static_cast<int>((a.N + bn - 1) / bn);
  p.num_tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
  p.band = band_tiles(a.M, a.N, a.K, p.num_m_tiles);
  if (wide && p.num_m_tiles >= 2 && duo_enabled())
    switch (duo_width(a.M, a.N, p.out_fp32 != 0)) {
      case 384: return launch_duo<384>(a, p, stream);
      case 192: return launch_duo<192>(a, p, stream);
      default: return launch_duo<256>(a, p, stream);
    }
  CUtensorMap ma, mb, mc;
  if (!make_map(&ma, a.A, 2, a.K, a.M, 1, BK, BM)) return MXFP8_ERR_CUDA;
  if (!make_out_map(&mc, a.C, a.M, a.N, 1, p.out_fp32 != 0, 3)) return MXFP8_ERR_CUDA;
  if (!make_map(&mb, a.B, 2, a.K, a.N, 1, BK, bn)) return MXFP8_ERR_CUDA;
  if (p.num_tiles > INT32_MAX) return MXFP8_ERR_INVALID_ARG;  // 32-bit tile arithmetic
  const int64_t grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
  return wide ? launch<256, kDense>(ma, mb, mc, p, grid, stream)
              : launch<128, kDense>(ma, mb, mc, p, grid, stream);
}

int launch_grouped_gemm(const GemmArgs& a, cudaStream_t stream) {
  if (a.num_experts > kMaxExperts) return MXFP8_ERR_INVALID_ARG;
  Params p{};
  p.sA = static_cast<const uint8_t*>(a.sA);
  p.sB = static_cast<const uint8_t*>(a.sB);
  p.C = a.C;
  p.out_fp32 = a.out_dtype == MXFP8_OUT_FP32;
  p.offsets = a.offsets;
  p.E = a.num_experts;
  p.total_rows = a.total_rows;
  p.status = a.status;
  p.wait_ns = wait_limit_ns();
  p.drain_ns = drain_limit_ns(p.wait_ns);
  CUtensorMap ma, mb, mc;
  if (a.op == MXFP8_OP_WGRAD) {
    // A = dY^T [N][T], B = X^T [K][T], C[e] = [N][K]
    p.M = a.N;
    p.N = a.K;
    p.K = a.total_rows;
    const bool wide = p.N > 128;
    const int bn = wide ? 256 : 128;
    p.num_m_tiles = static_cast<int>((p.M + BM - 1) / BM);
    p.num_n_tiles = static_cast<int>((p.N + bn - 1) / bn);
    const int64_t tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles * p.E;
    p.num_tiles = tiles;
    if (wide && p.num_m_tiles >= 2 && p.E <= kMaxDuoExperts && duo_enabled())
      return duo_grouped_width(kGroupWgrad, p.N, p.out_fp32 != 0) == 256
                 ? launch_duo_grouped<256, kGroupWgrad>(a, p, stream)
                 : launch_duo_grouped<192, kGroupWgrad>(a, p, stream);
    if (!make_map(&ma, a.A, 2, a.total_rows, p.M, 1, BK, BM)) return MXFP8_ERR_CUDA;
    if (!make_map(&mb, a.B, 2, a.total_rows, p.N, 1, BK, bn)) return MXFP8_ERR_CUDA;
    if (!make_out_map(&mc, a.C, p.M, p.N, p.E, p.out_fp32 != 0, 3)) return MXFP8_ERR_CUDA;
    if (tiles > INT32_MAX) return MXFP8_ERR_INVALID_ARG;  // 32-bit tile arithmetic
    const int64_t grid = tiles < num_sms() ? tiles : num_sms();
    return wide ? launch<256, kGroupWgrad>(ma, mb, mc, p, grid, stream)
                : launch<128, kGroupWgrad>(ma, mb, mc, p, grid, stream);
  }
  // fprop / dgrad: A [T][K] segmented by rows, B [E][N][K], C [T][N]
  p.M = a.total_rows;
  p.N = a.N;
  p.K = a.K;
  const bool wide = p.N > 128;
  const int bn = wide ? 256 : 128;
  const int64_t n_kt = (a.K + BK - 1) / BK;
  p.sb_item_bytes = ((a.N + 127) / 128) * n_kt * 512;
  p.num_m_tiles = static_cast<int>((a.total_rows + BM - 1) / BM + a.num_experts);
  p.num_n_tiles = static_cast<int>((p.N + bn - 1) / bn);
  const int64_t tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
  p.num_tiles = tiles;
  if (wide && p.E <= kMaxDuoExperts && duo_enabled())
    switch (duo_grouped_width(kGroupRows, p.N, p.out_fp32 != 0)) {
      case 384: return launch_duo_grouped<384, kGroupRows>(a, p, stream);
      case 192: return launch_duo_grouped<192, kGroupRows>(a, p, stream);
      default: return launch_duo_grouped<256, kGroupRows>(a, p, stream);
    }
  if (!make_map(&ma, a.A, 2, a.K, a.total_rows, 1, BK, BM)) return MXFP8_ERR_CUDA;
  if (!make_map(&mb, a.B, 3, a.K, a.N, a.num_experts, BK, bn)) return MXFP8_ERR_CUDA;
  if (!make_out_map(&mc, a.C, a.total_rows, p.N, 1, p.out_fp32 != 0, 3)) return MXFP8_ERR_CUDA;
  if (tiles > INT32_MAX) return MXFP8_ERR_INVALID_ARG;  // 32-bit tile arithmetic
  const int64_t grid = tiles < num_sms() ? tiles : num_sms();
  return wide ? launch<256, kGroupRows>(ma, mb, mc, p, grid, stream)
              : launch<128, kGroupRows>(ma, mb, mc, p, grid, stream);
}

}  // namespace mxfp8

// quantize.cu - MXFP8 quantizer kernels (row-wise and column-wise with a fused
// transpose), writing linear or tensor-core-swizzled E8M0 scales directly.
//
// Format: "End-to-End MXFP8 RL on Blackwell" (verl blog post), section "The pipeline",
// paragraph "The format" (E4M3 elements, blocks of 32, one power-of-two E8M0 scale per
// block); column-wise copies along tokens for the weight-gradient GEMM: the learner
// paragraph of the same section; scales written straight into the GEMM's layout instead
// of a separate rearrangement pass: section "Where the time goes".
//
// Each CTA owns a 128 x 128 BF16 tile (32 KB) and keeps all of it in flight at once.
// The row-wise kernel loads it into registers (eight 16-byte loads per thread, all issued
// before any is used). Kernels that write the column-wise copy copy it into shared memory
// with cp.async instead: no register is held while the loads are in flight, so six CTAs
// fit on an SM, and both copies read the tile from there. A 128 x 128 tile has exactly
// 128 x 4 blocks, i.e. one 512-byte swizzled scale tile, which the CTA assembles in
// shared memory and stores with 16-byte writes.
//
// Block maxima are taken two elements at once: max.NaN.xorsign.abs.bf16x2 in the MXFP8
// kernels (magnitudes compared, NaN wins; the sign bits are cleared once per block), and
// unsigned 16-bit maxima of the sign-cleared bits in the block-wise kernel, whose FP32
// scale needs the exact maximum even when it is subnormal.
//
// The block exponent is taken from the integer bits of the block's largest |BF16|
// (biased exponent E): scale byte = max(E - 8, 0) (floor(log2 amax) - 8, clamped at
// -127). Elements are scaled two at a time by 2^-e with one packed BF16 product (exact for a
// power-of-two scale), widened to FP32 and converted two at a time with
// cvt.rn.satfinite.e4m3x2 (round to nearest even, saturating). The dual kernel's row pass gives each thread one 32-element
// block and stores its 32 code bytes at once; the column pass reads column pairs from the
// shared tile, whose rows are padded so that both passes are free of bank conflicts.

#include <cstdint>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"
#include "mxfp8.h"

namespace mxfp8 {
namespace {

constexpr int kTile = 128;        // rows and columns of a CTA tile
constexpr int kThreads = 256;
constexpr int kTilePitch = kTile + 8;  // BF16 row pitch of the shared tile: 272 bytes
constexpr int kMaxExperts = 1024; // grouped calls: experts scanned in shared memory

// Expert segmentation of the token rows for grouped calls. Every CTA re-derives the
// prefix sums of ceil(count / 128) from the offsets, so that no table has to be kept in
// global memory; invalid offsets make every CTA return without writing anything.
struct Segments {
  int32_t off[kMaxExperts + 1];
  int32_t tile_base[kMaxExperts + 1];  // prefix sum of ceil(count_e / 128)
  int32_t warp_sum[kThreads / 32];     // scratch of the block-wide scan
  int ok;
};

// The prefix sums come from a block-wide scan: each thread sums the tile counts of
// kMaxExperts / kThreads consecutive experts, a warp shuffle scan and the warps' totals
// place each thread's run, and the thread writes its experts' bases. A grouped launch runs
// this in every CTA, so a serial loop over the experts by one thread would cost each CTA
// microseconds.
__device__ void load_segments(Segments& s, const int32_t* __restrict__ offsets, int E,
                              int64_t total_rows, int* status) {
  constexpr int kPer = kMaxExperts / kThreads;  // experts per thread
  static_assert(kPer * kThreads == kMaxExperts, "experts must split evenly over the CTA");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) s.ok = 1;
  __syncthreads();
  for (int i = t; i <= E; i += kThreads) s.off[i] = offsets[i];
  __syncthreads();
  int32_t tiles[kPer];
  int32_t mine = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = t * kPer + j;
    int32_t n = 0;
    if (e < E) {
      const int32_t lo = s.off[e], hi = s.off[e + 1];
      if (hi < lo || (lo & 31) || (hi & 31)) s.ok = 0;
      n = hi > lo ? (hi - lo + 127) / 128 : 0;
    }
    tiles[j] = n;
    mine += n;
  }
  if (t == 0 && (s.off[0] != 0 || static_cast<int64_t>(s.off[E]) != total_rows)) s.ok = 0;
  int32_t incl = mine;  // inclusive scan within the warp
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) s.warp_sum[warp] = incl;
  __syncthreads();
  int32_t base = incl - mine;
  for (int w = 0; w < warp; ++w) base += s.warp_sum[w];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = t * kPer + j;
    if (e < E) s.tile_base[e] = base;
    base += tiles[j];
  }
  if (t == kThreads - 1) s.tile_base[E] = base;  // the total: threads past E add nothing
  __syncthreads();
  if (t == 0 && !s.ok) latch_error(status, MXFP8_ERR_BAD_OFFSETS);
}

// Finds the expert owning global tile-row `t` (tile_base[e] <= t < tile_base[e+1]).
__device__ int find_expert(const Segments& s, int E, int t) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.tile_base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr uint32_t kAbs2 = 0x7FFF7FFFu;  // clears both BF16 sign bits of a word

// Per-half maximum of |a| and |b| for two BF16 pairs, NaN winning over every number; the
// sign bits of the result are meaningless (cleared by kAbs2 once per block). Compared with
// clearing both signs and taking an unsigned 16-bit maximum this is one instruction instead
// of three. A BF16 subnormal amax gives scale byte 0 whether or not it is flushed here.
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per-half unsigned 16-bit maximum of two words: on sign-cleared BF16 bits, the exact
// maximum magnitude, subnormals included (the block-wise FP32 scale depends on it).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 16 bytes global -> shared, bypassing L1; `valid` false writes 16 zero bytes instead.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16u : 0u) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}



// Scale byte from the largest |BF16| bits of a block; 0xFF for a NaN/Inf block.
// Floor rule (OCP): floor(log2 amax) - 8 = biased exponent - 135, byte = E - 8.
// Round-up rule: one more when the mantissa of amax exceeds 1.75 (amax > 448 * 2^e), so
// that nothing saturates. Both clamp at byte 0 (e = -127).
__device__ __forceinline__ uint32_t scale_byte(uint32_t amax_bits, int rule) {
  if (amax_bits >= 0x7F80u) return 0xFFu;
  int e = static_cast<int>(amax_bits >> 7) - 8;
  if (rule == MXFP8_RULE_CEIL) e += (amax_bits & 0x7Fu) > 0x60u;
  return e > 0 ? static_cast<uint32_t>(e) : 0u;
}

// 2^-e for scale byte s = e + 127, as an FP32 (a normal number for s <= 253; the 0xFF of a
// NaN/Inf block gives -Inf, whose products are discarded).
__device__ __forceinline__ float inv_scale(uint32_t s) {
  return __uint_as_float((254u - s) << 23);
}

// Two elements given as FP32 bit patterns (lo first in memory order) -> 2 bytes: each
// scaled by an IEEE single-precision product rounded to nearest (exact for a power-of-two
// scale), then one RNE-saturating E4M3 conversion of the pair. Two scalar products measured
// slightly faster than one packed mul.rn.f32x2 (whose operands must sit in a register pair).
__device__ __forceinline__ uint32_t e4m3x2_f32bits(uint32_t lo, uint32_t hi, float mul) {
  const float a = __fmul_rn(__uint_as_float(lo), mul);
  const float b = __fmul_rn(__uint_as_float(hi), mul);
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(b), "f"(a));
  return c;
}

// Two BF16 pairs (4 elements, memory order lo(w0), hi(w0), lo(w1), hi(w1)) -> 4 bytes.
// A BF16 value's FP32 bit pattern is its 16 bits shifted to the top half.
__device__ __forceinline__ uint32_t e4m3x4(uint32_t w0, uint32_t w1, float mul) {
  return e4m3x2_f32bits(w0 << 16, w0 & 0xFFFF0000u, mul) |
         (e4m3x2_f32bits(w1 << 16, w1 & 0xFFFF0000u, mul) << 16);
}

// The MXFP8 kernels scale by an exact power of two, so they can scale two BF16 values with
// one packed BF16 product (exact: the results lie in [2^-133, 2^9) or are far below E4M3's
// smallest subnormal, and BF16 keeps subnormals) before widening them for the conversion.
// The block-wise kernel's FP32 scale is not a power of two: it keeps the FP32 products.

// BF16 bits of 2^-e for scale byte s = e + 127 (a normal number for s <= 253; the 0xFF of a
// NaN/Inf block gives +Inf, whose products are discarded).
__device__ __forceinline__ uint32_t inv_scale_bf16(uint32_t s) { return ((254u - s) & 0xFFu) << 7; }

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two values given as FP32 bit patterns (lo first in memory order) -> 2 bytes, one
// RNE-saturating E4M3 conversion of the pair.
__device__ __forceinline__ uint32_t e4m3x2_of(uint32_t lo, uint32_t hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
      : "=h"(c) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
  return c;
}

// Two BF16 pairs (4 elements, memory order lo(w0), hi(w0), lo(w1), hi(w1)) scaled by the
// BF16 pair mul2 (2^-e in both halves) -> 4 bytes.
__device__ __forceinline__ uint32_t e4m3x4_pow2(uint32_t w0, uint32_t w1, uint32_t mul2) {
  const uint32_t v0 = mul_bf16x2(w0, mul2), v1 = mul_bf16x2(w1, mul2);
  return e4m3x2_of(v0 << 16, v0 & 0xFFFF0000u) | (e4m3x2_of(v1 << 16, v1 & 0xFFFF0000u) << 16);
}

// 32 bytes global store in one instruction (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&o)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"l"(p), "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]),
                 "r"(o[6]), "r"(o[7]) : "memory");
}

// The same 4 elements of a NaN/Inf block: 0x7F with each element's own sign. Blocks like
// this take a separate branch after the normal conversion, which stays free of selects.
__device__ __forceinline__ uint32_t nan4(uint32_t w0, uint32_t w1) {
  const uint32_t s0 = (w0 >> 8) & 0x80u, s1 = (w0 >> 24) & 0x80u;
  const uint32_t s2 = (w1 >> 8) & 0x80u, s3 = (w1 >> 24) & 0x80u;
  return (0x7Fu | s0) | ((0x7Fu | s1) << 8) | ((0x7Fu | s2) << 16) | ((0x7Fu | s3) << 24);
}

// One CTA = one 128 x 128 BF16 tile (128 token rows x 128 columns). kRow: write the
// row-wise copy (blocks along the columns); kCol: write the column-wise copy (blocks
// along the rows, emitted transposed). With both, the input is read once, into a shared
// tile whose rows are padded to 272 bytes: the row-wise pass (one thread per 32-block,
// eight consecutive rows per eight lanes) and the column-wise pass (one word per row and
// lane) then read it without bank conflicts.
struct QOut {
  uint8_t* codes;
  uint8_t* scales;
  int64_t scale_item_bytes;  // bytes of one batch item's scale block
};

// Jobs of a multi-tensor launch: job j owns the grid's tiles [tile_base[j], tile_base[j+1]).
struct QJobs {
  int n;
  const uint16_t* src[kMaxQuantizeJobs];
  int64_t rows[kMaxQuantizeJobs], cols[kMaxQuantizeJobs];
  uint8_t* out[kMaxQuantizeJobs];
  uint8_t* scales[kMaxQuantizeJobs];
  uint8_t* out_col[kMaxQuantizeJobs];
  uint8_t* scales_col[kMaxQuantizeJobs];
  int64_t tile_base[kMaxQuantizeJobs + 1];
};

// Row-wise copy of a 128 x 128 tile staged in shared memory: one thread per 32-block (8
// consecutive rows per 8 lanes, conflict-free with the padded pitch), 32 code bytes per
// thread; the scale bytes go to the 512-byte tile stile_r (swizzled) or straight out.
template <bool kSwizzled>
__device__ __forceinline__ void row_pass_smem(const uint16_t (*tile)[kTilePitch],
                                              uint8_t* stile_r, const QOut& ro, int64_t cols,
                                              int64_t row0, int rows_valid, int64_t col0,
                                              int cols_valid, int rule) {
  const int t = threadIdx.x;
  const int64_t s_cols = cols / 32;
  const int w = t >> 5, l = t & 31;
  const int b = l >> 3;
  const bool block_ok = 32 * b < cols_valid;
  const bool wide = (reinterpret_cast<uintptr_t>(ro.codes) & 31) == 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = 8 * w + (l & 7) + 64 * i;
    const uint4* rp = reinterpret_cast<const uint4*>(&tile[r][32 * b]);
    const uint4 x0 = rp[0], x1 = rp[1], x2 = rp[2], x3 = rp[3];
    uint32_t m2 = max_abs_bf16x2(
        max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(x0.x, x0.y), max_abs_bf16x2(x0.z, x0.w)),
                       max_abs_bf16x2(max_abs_bf16x2(x1.x, x1.y), max_abs_bf16x2(x1.z, x1.w))),
        max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(x2.x, x2.y), max_abs_bf16x2(x2.z, x2.w)),
                       max_abs_bf16x2(max_abs_bf16x2(x3.x, x3.y), max_abs_bf16x2(x3.z, x3.w))));
    m2 &= kAbs2;
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    const bool valid = block_ok && r < rows_valid;
    const uint32_t s = scale_byte(m, rule);
    if (valid) {
      uint32_t o[8];
      if (__builtin_expect(s != 0xFFu, 1)) {
        const uint32_t mul2 = inv_scale_bf16(s) * 0x10001u;
        o[0] = e4m3x4_pow2(x0.x, x0.y, mul2); o[1] = e4m3x4_pow2(x0.z, x0.w, mul2);
        o[2] = e4m3x4_pow2(x1.x, x1.y, mul2); o[3] = e4m3x4_pow2(x1.z, x1.w, mul2);
        o[4] = e4m3x4_pow2(x2.x, x2.y, mul2); o[5] = e4m3x4_pow2(x2.z, x2.w, mul2);
        o[6] = e4m3x4_pow2(x3.x, x3.y, mul2); o[7] = e4m3x4_pow2(x3.z, x3.w, mul2);
      } else {
        o[0] = nan4(x0.x, x0.y); o[1] = nan4(x0.z, x0.w);
        o[2] = nan4(x1.x, x1.y); o[3] = nan4(x1.z, x1.w);
        o[4] = nan4(x2.x, x2.y); o[5] = nan4(x2.z, x2.w);
        o[6] = nan4(x3.x, x3.y); o[7] = nan4(x3.z, x3.w);
      }
      uint8_t* dst = ro.codes + (row0 + r) * cols + col0 + 32 * b;
      if (wide) {
        st_global_v8(dst, o);
      } else {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    if (kSwizzled)
      stile_r[(r & 31) * 16 + (r >> 5) * 4 + b] = valid ? static_cast<uint8_t>(s) : 0;
    else if (valid)
      ro.scales[(row0 + r) * s_cols + col0 / 32 + b] = static_cast<uint8_t>(s);
  }
}

// Column-wise copy (transpose) of a 128 x 128 tile staged in shared memory; the tile
// buffer is reused to stage the transposed codes, so it is dead once this returns.
template <bool kSwizzled>
__device__ __forceinline__ void col_pass_smem(uint16_t (*tile)[kTilePitch], uint8_t* stile_c,
                                              const QOut& co, int64_t rows, int64_t row0,
                                              int rows_valid, int64_t col0, int cols_valid,
                                              int rule) {
  const int t = threadIdx.x;
  // thread = column pair (2cp, 2cp+1) x token block j (32 rows); each word read holds
  // both columns of one row (column c in the low half)
  const int w = t >> 5, lane = t & 31;
  const int cp = (w & 1) * 32 + lane;
  const int j = w >> 1;
  const int c = 2 * cp;
  const bool valid = c < cols_valid && 32 * j < rows_valid;
  const uint32_t* colw = reinterpret_cast<const uint32_t*>(&tile[32 * j][c]);
  constexpr int kRowWords = kTilePitch / 2;
  uint32_t m01 = 0;  // both columns' block maxima, one per half
#pragma unroll
  for (int i = 0; i < 32; ++i) m01 = max_abs_bf16x2(m01, colw[i * kRowWords]);
  m01 &= kAbs2;
  const uint32_t s0 = scale_byte(m01 & 0xFFFFu, rule), s1 = scale_byte(m01 >> 16, rule);
  uint4 stage_o0[2], stage_o1[2];
  if (valid) {
    uint32_t o0[8], o1[8];
    if (__builtin_expect(s0 != 0xFFu && s1 != 0xFFu, 1)) {
      // each row word holds column c (low half) and c + 1 (high half): one packed product
      // scales both by their own block's 2^-e
      const uint32_t mulp = inv_scale_bf16(s0) | (inv_scale_bf16(s1) << 16);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t b0 = mul_bf16x2(colw[(4 * q) * kRowWords], mulp);
        const uint32_t b1 = mul_bf16x2(colw[(4 * q + 1) * kRowWords], mulp);
        const uint32_t b2 = mul_bf16x2(colw[(4 * q + 2) * kRowWords], mulp);
        const uint32_t b3 = mul_bf16x2(colw[(4 * q + 3) * kRowWords], mulp);
        o0[q] = e4m3x2_of(b0 << 16, b1 << 16) | (e4m3x2_of(b2 << 16, b3 << 16) << 16);
        o1[q] = e4m3x2_of(b0 & 0xFFFF0000u, b1 & 0xFFFF0000u) |
                (e4m3x2_of(b2 & 0xFFFF0000u, b3 & 0xFFFF0000u) << 16);
      }
    } else {  // a NaN/Inf block in either column (rare)
      const float mul0 = inv_scale(s0), mul1 = inv_scale(s1);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t a0 = colw[(4 * q) * kRowWords], a1 = colw[(4 * q + 1) * kRowWords];
        const uint32_t a2 = colw[(4 * q + 2) * kRowWords], a3 = colw[(4 * q + 3) * kRowWords];
        const uint32_t c0a = __byte_perm(a0, a1, 0x5410), c0b = __byte_perm(a2, a3, 0x5410);
        const uint32_t c1a = __byte_perm(a0, a1, 0x7632), c1b = __byte_perm(a2, a3, 0x7632);
        o0[q] = s0 == 0xFFu ? nan4(c0a, c0b) : e4m3x4(c0a, c0b, mul0);
        o1[q] = s1 == 0xFFu ? nan4(c1a, c1b) : e4m3x4(c1a, c1b, mul1);
      }
    }
    stage_o0[0] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
    stage_o0[1] = make_uint4(o0[4], o0[5], o0[6], o0[7]);
    stage_o1[0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    stage_o1[1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
  }
  if (kSwizzled) {
    stile_c[(c & 31) * 16 + (c >> 5) * 4 + j] = valid ? static_cast<uint8_t>(s0) : 0;
    stile_c[((c + 1) & 31) * 16 + ((c + 1) >> 5) * 4 + j] = valid ? static_cast<uint8_t>(s1) : 0;
  } else if (valid) {
    const int64_t s_cols = rows / 32;
    co.scales[(col0 + c) * s_cols + row0 / 32 + j] = static_cast<uint8_t>(s0);
    co.scales[(col0 + c + 1) * s_cols + row0 / 32 + j] = static_cast<uint8_t>(s1);
  }
  // The transposed codes go through shared memory so that each output row's 128 bytes
  // leave in one coalesced piece: stage[row][chunk] holds 16-byte chunks, chunk index
  // XOR (row & 7) against bank conflicts; the BF16 tile buffer is reused once every
  // thread has read what it needs of it.
  __syncthreads();
  uint4* stage = reinterpret_cast<uint4*>(&tile[0][0]);
  if (valid) {
    stage[c * 8 + ((2 * j) ^ (c & 7))] = stage_o0[0];
    stage[c * 8 + ((2 * j + 1) ^ (c & 7))] = stage_o0[1];
    stage[(c + 1) * 8 + ((2 * j) ^ ((c + 1) & 7))] = stage_o1[0];
    stage[(c + 1) * 8 + ((2 * j + 1) ^ ((c + 1) & 7))] = stage_o1[1];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (t >> 3) + 32 * i;  // output row = tile column
    const int ch = t & 7;             // 16 tokens per chunk
    if (r < cols_valid && 16 * ch < rows_valid)
      *reinterpret_cast<uint4*>(co.codes + (col0 + r) * rows + row0 + 16 * ch) =
          stage[r * 8 + (ch ^ (r & 7))];
  }
}

template <bool kRow, bool kCol, bool kSwizzled, bool kGrouped, bool kMulti>
__global__ void __launch_bounds__(kThreads, kCol ? 6 : 1)
quantize_tile_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t cols, QOut ro,
                     QOut co, const int32_t* __restrict__ offsets, int E, int rule,
                     int* status, const QJobs jobs) {
  __shared__ __align__(16) uint16_t tile[kCol ? kTile : 1][kCol ? kTilePitch : 8];
  __shared__ __align__(16) uint8_t stile_r[512];
  __shared__ __align__(16) uint8_t stile_c[512];
  extern __shared__ __align__(16) uint8_t dyn[];  // Segments for grouped calls
  Segments* seg = reinterpret_cast<Segments*>(dyn);
  grid_dependency_wait();
  grid_launch_dependents();
  if (kGrouped) load_segments(*seg, offsets, E, rows, status);

  // ---- which tile, and where its two 512-byte scale tiles go
  int64_t bx = blockIdx.x, by = blockIdx.y, item = blockIdx.z;
  if constexpr (kMulti) {  // a 1-D grid over every job's tiles, job by job
    const int64_t g = blockIdx.x;
    int j = 0;
    while (j + 1 < jobs.n && g >= jobs.tile_base[j + 1]) ++j;
    src = jobs.src[j];
    rows = jobs.rows[j];
    cols = jobs.cols[j];
    ro = QOut{jobs.out[j], jobs.scales[j], 0};
    co = QOut{jobs.out_col[j], jobs.scales_col[j], 0};
    // tile counts are below 2^31 (checked on the host): 32-bit division, far cheaper than
    // the 64-bit one every thread would otherwise run
    const uint32_t local = static_cast<uint32_t>(g - jobs.tile_base[j]);
    const uint32_t n_ct = static_cast<uint32_t>((cols + kTile - 1) / kTile);
    by = local / n_ct;
    bx = local % n_ct;
    item = 0;
  }
  const int64_t n_col_tiles = (cols + kTile - 1) / kTile;  // = scale tiles per row-wise tile row
  int64_t row0, tile_row;       // first token row; global token-tile index
  int rows_valid;
  int64_t col_scale_tile;       // column-wise scale tile index
  if (!kGrouped) {
    tile_row = by;
    row0 = tile_row * kTile;
    const int64_t left = rows - row0;
    rows_valid = static_cast<int>(left < kTile ? left : kTile);
    col_scale_tile = bx * ((rows + kTile - 1) / kTile) + tile_row;
  } else {
    const int t = static_cast<int>(by);
    if (!seg->ok || t >= seg->tile_base[E]) return;
    const int e = find_expert(*seg, E, t);
    const int64_t i = t - seg->tile_base[e];
    tile_row = t;
    row0 = seg->off[e] + i * kTile;
    const int64_t left = seg->off[e + 1] - row0;
    rows_valid = static_cast<int>(left < kTile ? left : kTile);
    const int64_t cnt = seg->off[e + 1] - seg->off[e];
    col_scale_tile = n_col_tiles * seg->tile_base[e] +
                     bx * ((cnt + kTile - 1) / kTile) + i;
  }
  const int64_t row_scale_tile = tile_row * n_col_tiles + bx;

  src += item * rows * cols;
  if (kRow) {
    ro.codes += item * rows * cols;
    ro.scales += item * ro.scale_item_bytes;
  }
  if (kCol) {
    co.codes += item * rows * cols;
    co.scales += item * co.scale_item_bytes;
  }

  const int t = threadIdx.x;
  const int v = t & 15;             // 16-byte vector (8 elements) within the tile row
  const int rsub = t >> 4;          // rows rsub + 16 j
  const int64_t col0 = bx * kTile;
  const int64_t cols_left = cols - col0;
  const int cols_valid = static_cast<int>(cols_left < kTile ? cols_left : kTile);
  const bool col_ok = 8 * v < cols_valid;   // cols % 8 == 0 (% 32 == 0 with kRow)

  // ---- load the tile: into shared memory when a column-wise copy is made, else registers
  uint4 x[kCol ? 1 : 8];
  if constexpr (kCol) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = rsub + 16 * j;
      const bool ok = col_ok && r < rows_valid;
      cp_async16(&tile[r][8 * v], ok ? src + (row0 + r) * cols + col0 + 8 * v : src, ok);
    }
    cp_async_wait_all();
    __syncthreads();
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = rsub + 16 * j;
      if (col_ok && r < rows_valid)
        x[j] = ld_nc_v4(src + (row0 + r) * cols + col0 + 8 * v);
      else
        x[j] = make_uint4(0, 0, 0, 0);
    }
  }

  // ---- row-wise copy from the shared tile
  if constexpr (kRow && kCol)
    row_pass_smem<kSwizzled>(tile, stile_r, ro, cols, row0, rows_valid, col0, cols_valid, rule);

  // ---- row-wise copy from registers: the 4 lanes of a 32-block share amax
  if (kRow && !kCol) {
    const int64_t s_cols = cols / 32;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = rsub + 16 * j;
      const uint4 xv = x[j];
      uint32_t m2 = max_abs_bf16x2(max_abs_bf16x2(xv.x, xv.y), max_abs_bf16x2(xv.z, xv.w));
      m2 = max_abs_bf16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 1));
      m2 = max_abs_bf16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 2));
      m2 &= kAbs2;
      const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
      const bool valid = col_ok && r < rows_valid;
      const uint32_t s = scale_byte(m, rule);
      if (valid) {
        uint2 o;
        if (__builtin_expect(s != 0xFFu, 1)) {
          const uint32_t mul2 = inv_scale_bf16(s) * 0x10001u;
          o.x = e4m3x4_pow2(xv.x, xv.y, mul2);
          o.y = e4m3x4_pow2(xv.z, xv.w, mul2);
        } else {
          o.x = nan4(xv.x, xv.y);
          o.y = nan4(xv.z, xv.w);
        }
        *reinterpret_cast<uint2*>(ro.codes + (row0 + r) * cols + col0 + 8 * v) = o;
      }
      if ((v & 3) == 0) {
        const int b = v >> 2;  // block within the tile row
        if (kSwizzled)
          stile_r[(r & 31) * 16 + (r >> 5) * 4 + b] = valid ? static_cast<uint8_t>(s) : 0;
        else if (valid)
          ro.scales[(row0 + r) * s_cols + col0 / 32 + b] = static_cast<uint8_t>(s);
      }
    }
  }

  // ---- column-wise copy from the shared tile (transpose)
  if constexpr (kCol)
    col_pass_smem<kSwizzled>(tile, stile_c, co, rows, row0, rows_valid, col0, cols_valid, rule);

  // ---- the tile's swizzled scale tiles, 16 bytes per thread
  if (kSwizzled) {
    __syncthreads();
    if (kRow && t < 32)
      reinterpret_cast<uint4*>(ro.scales + row_scale_tile * 512)[t] =
          reinterpret_cast<const uint4*>(stile_r)[t];
    if (kCol && t >= 32 && t < 64)
      reinterpret_cast<uint4*>(co.scales + col_scale_tile * 512)[t - 32] =
          reinterpret_cast<const uint4*>(stile_c)[t - 32];
  }
}

// FP8 block-wise weight quantization: one FP32 (or power-of-two) scale per 128 x 128
// block ("End-to-End MXFP8 RL on Blackwell", section "A different grid, and drift"). One
// CTA per block: the block maximum comes from packed 16-bit maxima, warp shuffles and a
// shared-memory step; the factor s is 448 / amax (IEEE division, clamped to the largest
// float on overflow) or the power-of-two 2^-ceil(log2(amax / 448)); elements are
// E4M3(v * s) with the product rounded to single precision; 1 / s is stored.
// The scale choice is a run-time argument: one compiled kernel serves both (a separate
// power-of-two instantiation was scheduled with fewer loads in flight and ran 18% slower).
__global__ void __launch_bounds__(kThreads)
blockwise_quantize_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t cols,
                          uint8_t* __restrict__ out, float* __restrict__ scale_inv, int pow2) {
  __shared__ uint32_t warp_max[kThreads / 32];
  __shared__ float s_factor;
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = threadIdx.x, v = t & 15, rsub = t >> 4;
  const int64_t row0 = static_cast<int64_t>(blockIdx.y) * kTile;
  const int64_t col0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int rows_valid = static_cast<int>((rows - row0) < kTile ? (rows - row0) : kTile);
  const int cols_valid = static_cast<int>((cols - col0) < kTile ? (cols - col0) : kTile);
  const bool col_ok = 8 * v < cols_valid;  // cols % 8 == 0
  uint4 x[8];
  uint32_t m2 = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = rsub + 16 * j;
    x[j] = (col_ok && r < rows_valid) ? ld_nc_v4(src + (row0 + r) * cols + col0 + 8 * v)
                                      : make_uint4(0, 0, 0, 0);
    m2 = max_u16x2(m2, max_u16x2(max_u16x2(x[j].x & kAbs2, x[j].y & kAbs2),
                                 max_u16x2(x[j].z & kAbs2, x[j].w & kAbs2)));
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((t & 31) == 0) warp_max[t >> 5] = m;
  __syncthreads();
  if (t == 0) {
    uint32_t a = 0;
    for (int w = 0; w < kThreads / 32; ++w) a = max(a, warp_max[w]);
    float f, inv;
    if (a >= 0x7F80u) {                 // NaN or Inf in the block
      f = 0.f;
      inv = __uint_as_float(0x7FC00000u);
    } else if (a == 0) {                // all zero
      f = 1.f;
      inv = 1.f;
    } else if (pow2) {
      // e = ceil(log2(amax / 448)) >= -127; the BF16 exponent gives floor(log2 amax)
      int e = static_cast<int>(a >> 7) - 127 - 8 + ((a & 0x7Fu) > 0x60u ? 1 : 0);
      if ((a >> 7) == 0) e = -127;      // BF16 subnormal
      e = e < -127 ? -127 : e;
      f = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      inv = e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                      : __uint_as_float(0x00400000u);  // 2^-127
    } else {
      f = __fdiv_rn(448.f, __uint_as_float(a << 16));
      if (isinf(f)) f = 3.40282347e38f;  // the largest finite float
      inv = __fdiv_rn(1.f, f);
    }
    s_factor = f;
    scale_inv[static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x] = inv;
  }
  __syncthreads();
  const float f = s_factor;
  const bool nan_block = f == 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = rsub + 16 * j;
    if (!col_ok || r >= rows_valid) continue;
    uint2 o;
    if (!nan_block) {
      o.x = e4m3x4(x[j].x, x[j].y, f);
      o.y = e4m3x4(x[j].z, x[j].w, f);
    } else {
      o.x = nan4(x[j].x, x[j].y);
      o.y = nan4(x[j].z, x[j].w);
    }
    *reinterpret_cast<uint2*>(out + (row0 + r) * cols + col0 + 8 * v) = o;
  }
}

// One launch of kThreads-thread CTAs, with programmatic stream serialization unless it is
// turned off (the kernels wait for the previous kernel of the stream themselves).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, size_t dyn, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  return cudaLaunchKernelEx(&cfg, k, args...);
}

template <bool kRow, bool kCol, bool kSw, bool kGr>
cudaError_t launch_tiles(const QuantizeArgs& a, cudaStream_t stream) {
  const int64_t col_tiles = (a.cols + kTile - 1) / kTile;
  int64_t row_tiles = (a.rows + kTile - 1) / kTile;
  if (kGr) row_tiles += a.num_experts;  // upper bound: each expert adds one partial tile
  if (row_tiles > 65535 || col_tiles > 0x7FFFFFFF || a.batch > 65535)
    return cudaErrorInvalidValue;
  const size_t dyn = kGr ? sizeof(Segments) : 0;
  auto k = quantize_tile_kernel<kRow, kCol, kSw, kGr, false>;
  if (dyn) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(dyn));
    if (e != cudaSuccess) return e;
  }
  const QOut ro{static_cast<uint8_t*>(a.out), static_cast<uint8_t*>(a.scales),
                a.scale_item_bytes};
  const QOut co{static_cast<uint8_t*>(a.out_col), static_cast<uint8_t*>(a.scales_col),
                a.scale_item_bytes_col};
  const dim3 grid(static_cast<unsigned>(col_tiles), static_cast<unsigned>(row_tiles),
                 static_cast<unsigned>(a.batch));
  return launch_pdl(k, grid, dyn, stream, static_cast<const uint16_t*>(a.src), a.rows, a.cols,
                    ro, co, a.offsets, a.num_experts, a.rule, a.status, QJobs{});
}

template <bool kRow, bool kCol>
cudaError_t launch_axes(const QuantizeArgs& a, cudaStream_t stream) {
  if (a.offsets) return launch_tiles<kRow, kCol, true, true>(a, stream);
  if (a.layout == MXFP8_SCALES_SWIZZLED) return launch_tiles<kRow, kCol, true, false>(a, stream);
  return launch_tiles<kRow, kCol, false, false>(a, stream);
}

}  // namespace

int64_t scale_bytes_host(int64_t rows, int64_t cols, int axis, int layout);

cudaError_t launch_quantize_jobs(const QuantizeJobs& in, cudaStream_t stream) {
  QJobs j{};
  j.n = 0;
  int64_t tiles = 0;
  for (int i = 0; i < in.n; ++i) {
    if (in.rows[i] == 0 || in.cols[i] == 0) continue;
    const int n = j.n++;
    j.src[n] = static_cast<const uint16_t*>(in.src[i]);
    j.rows[n] = in.rows[i];
    j.cols[n] = in.cols[i];
    j.out[n] = static_cast<uint8_t*>(in.out[i]);
    j.scales[n] = static_cast<uint8_t*>(in.scales[i]);
    j.out_col[n] = static_cast<uint8_t*>(in.out_col[i]);
    j.scales_col[n] = static_cast<uint8_t*>(in.scales_col[i]);
    j.tile_base[n] = tiles;
    tiles += ((in.rows[i] + kTile - 1) / kTile) * ((in.cols[i] + kTile - 1) / kTile);
  }
  j.tile_base[j.n] = tiles;
  if (tiles == 0) return cudaSuccess;
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const QOut none{nullptr, nullptr, 0};
  const dim3 grid(static_cast<unsigned>(tiles));
  const uint16_t* no_src = nullptr;
  const int32_t* no_offsets = nullptr;
  if (in.layout == MXFP8_SCALES_SWIZZLED)
    return launch_pdl(quantize_tile_kernel<true, true, true, false, true>, grid, 0, stream,
                      no_src, int64_t{0}, int64_t{0}, none, none, no_offsets, 0,
                      int{MXFP8_RULE_FLOOR}, in.status, j);
  return launch_pdl(quantize_tile_kernel<true, true, false, false, true>, grid, 0, stream, no_src,
                    int64_t{0}, int64_t{0}, none, none, no_offsets, 0, int{MXFP8_RULE_FLOOR},
                    in.status, j);
}

cudaError_t launch_blockwise(const void* src, int64_t rows, int64_t cols, void* out,
                             float* scale_inv, bool pow2, cudaStream_t stream) {
  const int64_t gx = (cols + kTile - 1) / kTile, gy = (rows + kTile - 1) / kTile;
  if (gx == 0 || gy == 0) return cudaSuccess;
  if (gy > 65535 || gx > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  return launch_pdl(blockwise_quantize_kernel, grid, 0, stream,
                    static_cast<const uint16_t*>(src), rows, cols, static_cast<uint8_t*>(out),
                    scale_inv, pow2 ? 1 : 0);
}

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t stream) {
  if (a.rows == 0 || a.cols == 0 || a.batch == 0) return cudaSuccess;
  if (a.axis == kAxisBoth) return launch_axes<true, true>(a, stream);
  if (a.axis == MXFP8_AXIS_ROW) return launch_axes<true, false>(a, stream);
  return launch_axes<false, true>(a, stream);
}

}  // namespace mxfp8

// selfcheck.cu - post-synchronization self-check of quantized weights.
//
// "End-to-End MXFP8 RL on Blackwell" (verl blog post), section "Correctness: how it
// fails", the post-sync self-check (condition C3): after every synchronization one
// MXFP8 dense layer and one expert run through the MXFP8 kernel on random input and are
// compared with a BF16 GEMM on the dequantized synchronized weights. A healthy layer
// shows a relative error of a few percent (the cost of quantizing the activations); a
// stale or misplaced scale layout gives errors of order 1; the tolerance is 0.25.
//
// Here: X (BF16, random, caller-provided) is quantized and multiplied, by this library's
// own kernels, with the weight exactly as the GEMM reads it (E4M3 codes + swizzled
// scales: the derived layout) into an FP32 Y; a reference kernel recomputes every
// Y_ref[t][n] = sum_k x[t][k] * deq(W)[n][k] from the BF16 activations and the
// canonical synchronized weight (E4M3 codes + linear scales) with FP32 accumulation, and
// reduces ||Y - Y_ref||^2 and ||Y_ref||^2; a last kernel writes
// sqrt(||Y - Y_ref||^2 / ||Y_ref||^2). A derived layout that was not rebuilt from the
// synchronized weight therefore shows up as an error of order 1.

#include <cstdint>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"
#include "mxfp8.h"

namespace mxfp8 {
namespace {

constexpr int kRT = 32;   // reference tile: 32 tokens x 64 outputs per CTA
constexpr int kRN = 64;
constexpr int kRK = 32;   // one scale block of K per step

// E4M3 byte -> float, exact (hardware conversion through f16).
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  uint32_t h2;
  const uint16_t pair = static_cast<uint16_t>(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Block (t tile, n tile): Y_ref for a 32 x 64 tile, with the dequantized weight tile and
// the BF16 activations staged in shared memory, then its error terms added (double) to
// acc[0] (sum (y - y_ref)^2) and acc[1] (sum y_ref^2).
__global__ void __launch_bounds__(256)
selfcheck_ref_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ wq,
                     const uint8_t* __restrict__ ws, const float* __restrict__ y, int64_t T,
                     int64_t N, int64_t K, double* __restrict__ acc) {
  __shared__ float xs[kRT][kRK + 1];
  __shared__ float wsm[kRN][kRK + 1];
  __shared__ double red[2][8];
  const int tid = threadIdx.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kRT;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kRN;
  const int tt = tid / 16;         // 16 token rows of 2
  const int nn = tid % 16;         // 16 output cols of 4
  float sum[2][4] = {};
  const int64_t s_cols = K / 32;
  for (int64_t k0 = 0; k0 < K; k0 += kRK) {
    for (int i = tid; i < kRT * kRK; i += 256) {
      const int r = i / kRK, c = i % kRK;
      const int64_t t = t0 + r;
      xs[r][c] = t < T ? __uint_as_float(static_cast<uint32_t>(x[t * K + k0 + c]) << 16) : 0.f;
    }
    for (int i = tid; i < kRN * kRK; i += 256) {
      const int r = i / kRK, c = i % kRK;
      const int64_t n = n0 + r;
      float v = 0.f;
      if (n < N) {
        const uint32_t sb = ws[n * s_cols + k0 / 32];  // linear scales
        v = e4m3_to_float(wq[n * K + k0 + c]) * exp2f(static_cast<float>(static_cast<int>(sb) - 127));
      }
      wsm[r][c] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      const float a0 = xs[2 * tt][kk], a1 = xs[2 * tt + 1][kk];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float b = wsm[4 * nn + j][kk];
        sum[0][j] = fmaf(a0, b, sum[0][j]);
        sum[1][j] = fmaf(a1, b, sum[1][j]);
      }
    }
    __syncthreads();
  }
  double e2 = 0.0, r2 = 0.0;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t t = t0 + 2 * tt + i, n = n0 + 4 * nn + j;
      if (t < T && n < N) {
        const double ref = sum[i][j];
        const double d = static_cast<double>(y[t * N + n]) - ref;
        e2 += d * d;
        r2 += ref * ref;
      }
    }
  for (int o = 16; o > 0; o >>= 1) {
    e2 += __shfl_xor_sync(0xFFFFFFFFu, e2, o);
    r2 += __shfl_xor_sync(0xFFFFFFFFu, r2, o);
  }
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = e2;
    red[1][tid >> 5] = r2;
  }
  __syncthreads();
  if (tid == 0) {
    double a = 0.0, b = 0.0;
    for (int w = 0; w < 8; ++w) {
      a += red[0][w];
      b += red[1][w];
    }
    atomicAdd(&acc[0], a);
    atomicAdd(&acc[1], b);
  }
}

__global__ void selfcheck_finish_kernel(const double* __restrict__ acc, float* __restrict__ out) {
  out[0] = acc[1] > 0.0 ? static_cast<float>(sqrt(acc[0] / acc[1])) : (acc[0] > 0.0 ? INFINITY : 0.f);
}

// Workspace of the allocation-free self-check (mxfp8_selfcheck_noalloc): a fixed array
// in this module, present on every device that loads the library until the process
// exits. All calls share it.
static __device__ __align__(256) uint8_t g_selfcheck_scratch[kSelfcheckNoallocMaxBytes];

}  // namespace

int64_t selfcheck_workspace_bytes(int64_t T, int64_t N, int64_t K) {
  // Each term is formed with overflow checks: T, N and K may each be near 2^31, so their
  // products can leave int64. Any overflow makes the size invalid (-1), which every caller
  // rejects, so no size can wrap around to a small value that passes a capacity check.
  if (T <= 0 || N <= 0 || K <= 0) return -1;
  int64_t tk, tn, tn4, xs_tiles, xs, sum;
  if (__builtin_mul_overflow(T, K, &tk) || __builtin_mul_overflow(T, N, &tn) ||
      __builtin_mul_overflow(tn, int64_t(4), &tn4) ||
      __builtin_mul_overflow((T + 127) / 128, (K / 32 + 3) / 4, &xs_tiles) ||
      __builtin_mul_overflow(xs_tiles, int64_t(512), &xs))
    return -1;
  constexpr int64_t kPad = 255;  // each part is rounded up to 256 bytes
  if (tk > INT64_MAX / 4 || tn4 > INT64_MAX / 4 || xs > INT64_MAX / 4) return -1;
  auto up = [](int64_t b) { return (b + kPad) / 256 * 256; };
  if (__builtin_add_overflow(up(tk), up(xs), &sum) || __builtin_add_overflow(sum, up(tn4), &sum) ||
      __builtin_add_overflow(sum, int64_t(256), &sum))
    return -1;
  return sum;
}

int launch_selfcheck(const SelfcheckArgs& a, cudaStream_t stream) {
  auto up = [](int64_t b) { return (b + 255) / 256 * 256; };
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  uint8_t* xq = ws;
  uint8_t* xsc = xq + up(a.T * a.K);
  float* y = reinterpret_cast<float*>(xsc + up(((a.T + 127) / 128) * ((a.K / 32 + 3) / 4) * 512));
  double* acc = reinterpret_cast<double*>(reinterpret_cast<uint8_t*>(y) + up(a.T * a.N * 4));

  QuantizeArgs q{};
  q.src = a.x;
  q.batch = 1;
  q.rows = a.T;
  q.cols = a.K;
  q.axis = MXFP8_AXIS_ROW;
  q.out = xq;
  q.scales = xsc;
  q.layout = MXFP8_SCALES_SWIZZLED;
  q.status = a.status;
  if (launch_quantize(q, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  GemmArgs g{xq, xsc, a.w_codes, a.w_scales, y, a.T, a.N, a.K, MXFP8_OP_FPROP, MXFP8_OUT_FP32,
             nullptr, 0, 0, a.status};
  const int st = launch_gemm(g, stream);
  if (st != MXFP8_OK) return st;
  if (cudaMemsetAsync(acc, 0, 2 * sizeof(double), stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  // launched with cudaLaunchKernelEx, whose return value is this launch's own status (an
  // error left pending by an unrelated earlier call is not reported as this one's)
  const dim3 grid(static_cast<unsigned>((a.N + kRN - 1) / kRN),
                  static_cast<unsigned>((a.T + kRT - 1) / kRT));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  if (cudaLaunchKernelEx(&cfg, selfcheck_ref_kernel, static_cast<const uint16_t*>(a.x),
                         static_cast<const uint8_t*>(a.ref_codes),
                         static_cast<const uint8_t*>(a.ref_scales), static_cast<const float*>(y),
                         a.T, a.N, a.K, acc) != cudaSuccess)
    return MXFP8_ERR_CUDA;
  cudaLaunchConfig_t one = {};
  one.gridDim = dim3(1, 1, 1);
  one.blockDim = dim3(1, 1, 1);
  one.stream = stream;
  return cudaLaunchKernelEx(&one, selfcheck_finish_kernel, static_cast<const double*>(acc),
                            a.rel_err) == cudaSuccess
             ? MXFP8_OK
             : MXFP8_ERR_CUDA;
}

}  // namespace mxfp8

namespace mxfp8 {

// Device address of the fixed workspace, looked up once per device with that device
// current (host code must not use the array's name as a device address). The per-device
// cache is guarded by a mutex, so host threads that make their first calls at the same
// time do not race on it.
int selfcheck_noalloc_workspace(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MXFP8_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_selfcheck_scratch) != cudaSuccess || p == nullptr)
      return MXFP8_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return MXFP8_OK;
}

}  // namespace mxfp8

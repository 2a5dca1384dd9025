// api.cu - the extern "C" boundary (include/mxfp8.h): argument checks, per-device
// set-up (architecture check, SM count, status word) and dispatch to the launchers.

#include <cstdint>
#include <cstdlib>
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "mxfp8.h"

namespace mxfp8 {

namespace {

// First error a kernel detected on this device since the host last read it.
__device__ int g_device_status;

// mxfp8_get_device_status takes the word with one atomic exchange on the device, so an
// error latched by a kernel on another stream is either taken by this read or left for the
// next one, never cleared unread. Each call gets its own slot for the taken value, so that
// calls from several host threads do not overwrite each other's result. Slots are handed out
// round robin, so only more than 64 reads in flight at once could share one.
constexpr unsigned kStatusSlots = 64;
__device__ int g_status_taken[kStatusSlots];
std::atomic<unsigned> g_status_slot{0};

__global__ void take_status_kernel(unsigned slot) {
  g_status_taken[slot] = atomicExch(&g_device_status, 0);
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  // set up once per device under g_mu; `ready` is published last (release) and read first
  // (acquire), so a caller that sees it set also sees the fields below
  std::atomic<bool> ready{false};
  bool supported = false;
  int sms = 0;
  int* status = nullptr;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Per-device set-up on first use: capability 10.3 (GB300) required, SM count cached,
// address of the status word looked up. Returns MXFP8_OK or an error code.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MXFP8_ERR_CUDA;
  DeviceState& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int major = 0, minor = 0, sms = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MXFP8_ERR_CUDA;
      d.supported = (major == 10 && minor == 3);
      d.sms = sms;
      if (d.supported) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return MXFP8_ERR_CUDA;
        d.status = static_cast<int*>(p);
      }
      d.ready.store(true, std::memory_order_release);
    }
  }
  if (!d.supported) return MXFP8_ERR_UNSUPPORTED_ARCH;
  *out = &d;
  return MXFP8_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// a * b * c into *out, false if the product leaves int64 (sizes of impossible tensors).
bool mul3(int64_t a, int64_t b, int64_t c, int64_t* out) {
  int64_t ab = 0;
  return !__builtin_mul_overflow(a, b, &ab) && !__builtin_mul_overflow(ab, c, out);
}

constexpr int64_t kMaxTokenTiles = 65535;  // grid.y limit of the quantizer launch
// grid.y limit of the self-check's reference kernel (32 tokens per CTA row)
constexpr int64_t kMaxSelfcheckTokens = int64_t(32) * 65535;

}  // namespace

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  return (dev >= 0 && dev < kMaxDevices && g_dev[dev].sms > 0) ? g_dev[dev].sms : 148;
}

int64_t scale_bytes_host(int64_t rows, int64_t cols, int axis, int layout) {
  if (rows < 0 || cols < 0 || rows > INT64_MAX - 127 || cols > INT64_MAX - 127) return -1;
  int64_t s_rows, s_cols;
  if (axis == MXFP8_AXIS_ROW) {
    if (cols % 32) return -1;
    s_rows = rows;
    s_cols = cols / 32;
  } else if (axis == MXFP8_AXIS_COL) {
    if (rows % 32) return -1;
    s_rows = cols;
    s_cols = rows / 32;
  } else {
    return -1;
  }
  int64_t bytes = 0;
  if (layout == MXFP8_SCALES_LINEAR) return mul3(s_rows, s_cols, 1, &bytes) ? bytes : -1;
  if (layout == MXFP8_SCALES_SWIZZLED) {
    if (s_rows == 0 || s_cols == 0) return 0;
    return mul3(cdiv(s_rows, 128), cdiv(s_cols, 4), 512, &bytes) ? bytes : -1;
  }
  return -1;
}

}  // namespace mxfp8

using namespace mxfp8;

extern "C" {

int mxfp8_version(void) { return MXFP8_ABI_VERSION; }

const char* mxfp8_status_string(int status) {
  switch (status) {
    case MXFP8_OK: return "ok";
    case MXFP8_ERR_INVALID_ARG: return "invalid argument";
    case MXFP8_ERR_ALIGNMENT: return "alignment: blocked dim not a multiple of 32 or pointer not 16-byte aligned";
    case MXFP8_ERR_UNSUPPORTED_ARCH: return "unsupported device (needs compute capability 10.3, sm_103a)";
    case MXFP8_ERR_CUDA: return "CUDA call failed";
    case MXFP8_ERR_BAD_OFFSETS: return "expert offsets invalid (must be 0-based, non-decreasing, 32-aligned, end at total_rows)";
    case MXFP8_ERR_TIMEOUT: return "a kernel pipeline wait timed out; its work was abandoned";
    default: return "unknown status";
  }
}

size_t mxfp8_scale_bytes(int64_t rows, int64_t cols, int axis, int scale_layout) {
  const int64_t b = scale_bytes_host(rows, cols, axis, scale_layout);
  return b < 0 ? 0 : static_cast<size_t>(b);
}

size_t mxfp8_grouped_scale_bytes(int64_t total_rows, int64_t cols, int num_experts, int axis) {
  if (total_rows < 0 || cols <= 0 || num_experts <= 0 || total_rows % 32) return 0;
  if (total_rows > INT64_MAX - 127) return 0;
  int64_t bytes = 0;
  const int64_t tiles = cdiv(total_rows, 128) + num_experts;  // bound on sum of ceil(count / 128)
  if (axis == MXFP8_AXIS_ROW) {
    if (cols % 32) return 0;
    return mul3(tiles, cdiv(cols / 32, 4), 512, &bytes) ? static_cast<size_t>(bytes) : 0;
  }
  if (axis == MXFP8_AXIS_COL)
    return mul3(cdiv(cols, 128), tiles, 512, &bytes) ? static_cast<size_t>(bytes) : 0;
  return 0;
}

// axis: MXFP8_AXIS_ROW, MXFP8_AXIS_COL or kAxisBoth (out/scales = row-wise copy,
// out2/scales2 = column-wise copy).
static int quantize_common(const void* src, int64_t batch, int64_t rows, int64_t cols, int axis,
                           void* out, void* scales, void* out2, void* scales2, int layout,
                           const int32_t* offsets, int E, void* stream,
                           int rule = MXFP8_RULE_FLOOR) {
  if (rule != MXFP8_RULE_FLOOR && rule != MXFP8_RULE_CEIL) return MXFP8_ERR_INVALID_ARG;
  if (batch < 0 || rows < 0 || cols < 0) return MXFP8_ERR_INVALID_ARG;
  if (axis != MXFP8_AXIS_ROW && axis != MXFP8_AXIS_COL && axis != kAxisBoth)
    return MXFP8_ERR_INVALID_ARG;
  if (layout != MXFP8_SCALES_LINEAR && layout != MXFP8_SCALES_SWIZZLED)
    return MXFP8_ERR_INVALID_ARG;
  const bool row = axis != MXFP8_AXIS_COL, col = axis != MXFP8_AXIS_ROW;
  if (row && cols % 32) return MXFP8_ERR_ALIGNMENT;
  if (col && (rows % 32 || cols % 8)) return MXFP8_ERR_ALIGNMENT;
  if (batch == 0 || rows == 0 || cols == 0) return MXFP8_OK;
  int64_t elems = 0;  // BF16 input bytes = 2 * elems; the kernels index in int64
  if (!mul3(batch, rows, cols, &elems) || elems > INT64_MAX / 2) return MXFP8_ERR_INVALID_ARG;
  if (!src || !out || !scales) return MXFP8_ERR_INVALID_ARG;
  if (axis == kAxisBoth && (!out2 || !scales2)) return MXFP8_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(out) || (out2 && !aligned16(out2)))
    return MXFP8_ERR_ALIGNMENT;
  if (layout == MXFP8_SCALES_SWIZZLED && (!aligned16(scales) || (scales2 && !aligned16(scales2))))
    return MXFP8_ERR_ALIGNMENT;
  if (batch > 65535) return MXFP8_ERR_INVALID_ARG;
  const int64_t token_tiles = cdiv(rows, 128) + (offsets ? E : 0);
  if (token_tiles > kMaxTokenTiles || cdiv(cols, 128) > 0x7FFFFFFF) return MXFP8_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  const int st = device_state(&d);
  if (st != MXFP8_OK) return st;
  QuantizeArgs a{};
  a.src = src;
  a.batch = batch;
  a.rows = rows;
  a.cols = cols;
  a.axis = axis;
  a.layout = layout;
  a.offsets = offsets;
  a.num_experts = E;
  a.rule = rule;
  a.status = d->status;
  if (row) {
    a.out = out;
    a.scales = scales;
    a.scale_item_bytes = scale_bytes_host(rows, cols, MXFP8_AXIS_ROW, layout);
  }
  if (col) {
    a.out_col = axis == kAxisBoth ? out2 : out;
    a.scales_col = axis == kAxisBoth ? scales2 : scales;
    a.scale_item_bytes_col = scale_bytes_host(rows, cols, MXFP8_AXIS_COL, layout);
  }
  return launch_quantize(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MXFP8_OK
                                                                               : MXFP8_ERR_CUDA;
}

int mxfp8_quantize(const void* src_dev, int64_t rows, int64_t cols, int axis, void* out_dev,
                   void* scales_dev, int scale_layout, void* stream) {
  if (axis != MXFP8_AXIS_ROW && axis != MXFP8_AXIS_COL) return MXFP8_ERR_INVALID_ARG;
  return quantize_common(src_dev, 1, rows, cols, axis, out_dev, scales_dev, nullptr, nullptr,
                         scale_layout, nullptr, 0, stream);
}

int mxfp8_quantize_rule(const void* src_dev, int64_t rows, int64_t cols, int axis,
                        void* out_dev, void* scales_dev, int scale_layout, int scale_rule,
                        void* stream) {
  if (axis != MXFP8_AXIS_ROW && axis != MXFP8_AXIS_COL) return MXFP8_ERR_INVALID_ARG;
  return quantize_common(src_dev, 1, rows, cols, axis, out_dev, scales_dev, nullptr, nullptr,
                         scale_layout, nullptr, 0, stream, scale_rule);
}

int mxfp8_quantize_dual(const void* src_dev, int64_t rows, int64_t cols, void* row_out_dev,
                        void* row_scales_dev, void* col_out_dev, void* col_scales_dev,
                        int scale_layout, void* stream) {
  return quantize_common(src_dev, 1, rows, cols, kAxisBoth, row_out_dev, row_scales_dev,
                         col_out_dev, col_scales_dev, scale_layout, nullptr, 0, stream);
}

int mxfp8_quantize_dual_multi(const mxfp8_dual_job* jobs, int num_jobs, int scale_layout,
                              void* stream) {
  if (!jobs || num_jobs < 1 || num_jobs > MXFP8_MAX_DUAL_JOBS) return MXFP8_ERR_INVALID_ARG;
  if (scale_layout != MXFP8_SCALES_LINEAR && scale_layout != MXFP8_SCALES_SWIZZLED)
    return MXFP8_ERR_INVALID_ARG;
  static_assert(MXFP8_MAX_DUAL_JOBS <= kMaxQuantizeJobs, "job table too small");
  QuantizeJobs q{};
  q.n = num_jobs;
  q.layout = scale_layout;
  int64_t tiles = 0;
  for (int i = 0; i < num_jobs; ++i) {
    const mxfp8_dual_job& j = jobs[i];
    // the same checks as mxfp8_quantize_dual
    if (j.rows < 0 || j.cols < 0) return MXFP8_ERR_INVALID_ARG;
    if (j.rows % 32 || j.cols % 32) return MXFP8_ERR_ALIGNMENT;
    if (j.rows == 0 || j.cols == 0) continue;
    if (!j.src || !j.row_out || !j.row_scales || !j.col_out || !j.col_scales)
      return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(j.src) || !aligned16(j.row_out) || !aligned16(j.col_out))
      return MXFP8_ERR_ALIGNMENT;
    if (scale_layout == MXFP8_SCALES_SWIZZLED &&
        (!aligned16(j.row_scales) || !aligned16(j.col_scales)))
      return MXFP8_ERR_ALIGNMENT;
    if (cdiv(j.rows, 128) > kMaxTokenTiles || cdiv(j.cols, 128) > 0x7FFFFFFF)
      return MXFP8_ERR_INVALID_ARG;
    tiles += cdiv(j.rows, 128) * cdiv(j.cols, 128);
    q.src[i] = j.src;
    q.rows[i] = j.rows;
    q.cols[i] = j.cols;
    q.out[i] = j.row_out;
    q.scales[i] = j.row_scales;
    q.out_col[i] = j.col_out;
    q.scales_col[i] = j.col_scales;
  }
  if (tiles > 0x7FFFFFFF) return MXFP8_ERR_INVALID_ARG;
  if (tiles == 0) return MXFP8_OK;
  DeviceState* d = nullptr;
  const int st = device_state(&d);
  if (st != MXFP8_OK) return st;
  q.status = d->status;
  return launch_quantize_jobs(q, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MXFP8_OK
             : MXFP8_ERR_CUDA;
}

size_t mxfp8_blockwise_scale_count(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % 8) return 0;
  if (rows > INT64_MAX - 127 || cols > INT64_MAX - 127) return 0;
  int64_t n = 0;
  return mul3(cdiv(rows, 128), cdiv(cols, 128), 1, &n) ? static_cast<size_t>(n) : 0;
}

int mxfp8_quantize_blockwise(const void* src_dev, int64_t rows, int64_t cols, void* out_dev,
                             float* scale_inv_dev, int scale_type, void* stream) {
  if (scale_type != MXFP8_BW_SCALE_FP32 && scale_type != MXFP8_BW_SCALE_POW2)
    return MXFP8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0) return MXFP8_ERR_INVALID_ARG;
  if (cols % 8) return MXFP8_ERR_ALIGNMENT;
  if (rows == 0 || cols == 0) return MXFP8_OK;
  if (!src_dev || !out_dev || !scale_inv_dev) return MXFP8_ERR_INVALID_ARG;
  if (!aligned16(src_dev) || !aligned16(out_dev) ||
      (reinterpret_cast<uintptr_t>(scale_inv_dev) & 3u))
    return MXFP8_ERR_ALIGNMENT;
  if (cdiv(rows, 128) > 65535 || cdiv(cols, 128) > 0x7FFFFFFF) return MXFP8_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  const int st = device_state(&d);
  if (st != MXFP8_OK) return st;
  return launch_blockwise(src_dev, rows, cols, out_dev, scale_inv_dev,
                          scale_type == MXFP8_BW_SCALE_POW2,
                          static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MXFP8_OK
             : MXFP8_ERR_CUDA;
}

int mxfp8_quantize_batched(const void* src_dev, int64_t batch, int64_t rows, int64_t cols,
                           int axis, void* out_dev, void* scales_dev, int scale_layout,
                           void* stream) {
  if (axis != MXFP8_AXIS_ROW && axis != MXFP8_AXIS_COL) return MXFP8_ERR_INVALID_ARG;
  return quantize_common(src_dev, batch, rows, cols, axis, out_dev, scales_dev, nullptr, nullptr,
                         scale_layout, nullptr, 0, stream);
}

int mxfp8_quantize_grouped(const void* src_dev, int64_t total_rows, int64_t cols, int axis,
                           const int32_t* expert_offsets_dev, int num_experts, void* out_dev,
                           void* scales_dev, void* stream) {
  if (num_experts <= 0 || num_experts > 1024 || !expert_offsets_dev) return MXFP8_ERR_INVALID_ARG;
  if (axis != MXFP8_AXIS_ROW && axis != MXFP8_AXIS_COL) return MXFP8_ERR_INVALID_ARG;
  if (total_rows % 32) return MXFP8_ERR_ALIGNMENT;
  return quantize_common(src_dev, 1, total_rows, cols, axis, out_dev, scales_dev, nullptr,
                         nullptr, MXFP8_SCALES_SWIZZLED, expert_offsets_dev, num_experts, stream);
}

int mxfp8_quantize_grouped_dual(const void* src_dev, int64_t total_rows, int64_t cols,
                                const int32_t* expert_offsets_dev, int num_experts,
                                void* row_out_dev, void* row_scales_dev, void* col_out_dev,
                                void* col_scales_dev, void* stream) {
  if (num_experts <= 0 || num_experts > 1024 || !expert_offsets_dev) return MXFP8_ERR_INVALID_ARG;
  if (total_rows % 32) return MXFP8_ERR_ALIGNMENT;
  return quantize_common(src_dev, 1, total_rows, cols, kAxisBoth, row_out_dev, row_scales_dev,
                         col_out_dev, col_scales_dev, MXFP8_SCALES_SWIZZLED, expert_offsets_dev,
                         num_experts, stream);
}

// C = 0 for a reduction over nothing (K = 0, or no tokens for a grouped wgrad): `elems`
// output elements zero-filled on the stream; C must be valid and 16-byte aligned.
static int zero_fill_output(void* C, int64_t elems, int out_dtype, void* stream) {
  if (!C) return MXFP8_ERR_INVALID_ARG;
  if (!aligned16(C)) return MXFP8_ERR_ALIGNMENT;
  int64_t bytes = 0;
  if (!mul3(elems, out_dtype == MXFP8_OUT_FP32 ? 4 : 2, 1, &bytes)) return MXFP8_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  const int st = device_state(&d);
  if (st != MXFP8_OK) return st;
  return cudaMemsetAsync(C, 0, static_cast<size_t>(bytes), static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MXFP8_OK
             : MXFP8_ERR_CUDA;
}

static int gemm_checks(const void* A, const void* sA, const void* B, const void* sB, void* C,
                       int op, int out_dtype) {
  if (!A || !sA || !B || !sB || !C) return MXFP8_ERR_INVALID_ARG;
  if (op < MXFP8_OP_FPROP || op > MXFP8_OP_WGRAD) return MXFP8_ERR_INVALID_ARG;
  if (out_dtype != MXFP8_OUT_BF16 && out_dtype != MXFP8_OUT_FP32) return MXFP8_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(C))
    return MXFP8_ERR_ALIGNMENT;
  return MXFP8_OK;
}

int mxfp8_gemm(const void* A_dev, const void* sA_dev, const void* B_dev, const void* sB_dev,
               void* C_dev, int64_t M, int64_t N, int64_t K, int op, int out_dtype,
               void* stream) {
  return mxfp8_gemm_ws(A_dev, sA_dev, B_dev, sB_dev, C_dev, M, N, K, op, out_dtype, nullptr,
                       0, stream);
}

size_t mxfp8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int op, int out_dtype) {
  if (M <= 0 || N <= 0 || K <= 0 || M > 0x7FFFFF00 || N > 0x7FFFFF00 || K > 0x7FFFFF00)
    return 0;
  if (op < MXFP8_OP_FPROP || op > MXFP8_OP_WGRAD) return 0;
  if (out_dtype != MXFP8_OUT_BF16 && out_dtype != MXFP8_OUT_FP32) return 0;
  DeviceState* d = nullptr;
  if (device_state(&d) != MXFP8_OK) return 0;
  return gemm_workspace_bytes(M, N, K, out_dtype);
}

int mxfp8_gemm_ws(const void* A_dev, const void* sA_dev, const void* B_dev, const void* sB_dev,
                  void* C_dev, int64_t M, int64_t N, int64_t K, int op, int out_dtype,
                  void* workspace_dev, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return MXFP8_ERR_INVALID_ARG;
  if (M > 0x7FFFFF00 || N > 0x7FFFFF00 || K > 0x7FFFFF00) return MXFP8_ERR_INVALID_ARG;
  if (K % 32 || M % 16 || N % 16) return MXFP8_ERR_ALIGNMENT;
  if (op < MXFP8_OP_FPROP || op > MXFP8_OP_WGRAD) return MXFP8_ERR_INVALID_ARG;
  if (out_dtype != MXFP8_OUT_BF16 && out_dtype != MXFP8_OUT_FP32) return MXFP8_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MXFP8_OK;  // an empty output: nothing to read or write
  if (K == 0) return zero_fill_output(C_dev, M * N, out_dtype, stream);  // the empty sum
  int st = gemm_checks(A_dev, sA_dev, B_dev, sB_dev, C_dev, op, out_dtype);
  if (st != MXFP8_OK) return st;
  if (workspace_dev && (reinterpret_cast<uintptr_t>(workspace_dev) & 31))
    return MXFP8_ERR_ALIGNMENT;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != MXFP8_OK) return st;
  GemmArgs a{A_dev, sA_dev, B_dev, sB_dev, C_dev, M, N, K, op, out_dtype, nullptr, 0, 0,
             d->status, workspace_dev, workspace_dev ? workspace_bytes : 0};
  return launch_gemm(a, static_cast<cudaStream_t>(stream));
}

int mxfp8_grouped_gemm(const void* A_dev, const void* sA_dev, const void* B_dev,
                       const void* sB_dev, void* C_dev, const int32_t* expert_offsets_dev,
                       int num_experts, int64_t total_rows, int64_t N, int64_t K, int op,
                       int out_dtype, void* stream) {
  if (num_experts <= 0 || num_experts > 1024 || !expert_offsets_dev) return MXFP8_ERR_INVALID_ARG;
  if (total_rows < 0 || N < 0 || K < 0) return MXFP8_ERR_INVALID_ARG;
  if (total_rows > 0x7FFFFF00 || N > 0x7FFFFF00 || K > 0x7FFFFF00) return MXFP8_ERR_INVALID_ARG;
  if (total_rows % 32 || K % 32 || N % 16) return MXFP8_ERR_ALIGNMENT;
  if (op < MXFP8_OP_FPROP || op > MXFP8_OP_WGRAD) return MXFP8_ERR_INVALID_ARG;
  if (out_dtype != MXFP8_OUT_BF16 && out_dtype != MXFP8_OUT_FP32) return MXFP8_ERR_INVALID_ARG;
  // Empty cases read no operand, so A, B and their scales may then be empty (NULL), and the
  // offsets are not read: an empty output (N = 0, K = 0 for wgrad, no tokens for fprop and
  // dgrad) is a no-op; a reduction over nothing (no tokens for wgrad, K = 0 for fprop and
  // dgrad) zero-fills C.
  const bool wgrad = op == MXFP8_OP_WGRAD;
  if (N == 0 || (wgrad ? K == 0 : total_rows == 0)) return MXFP8_OK;
  if (wgrad && total_rows == 0) {
    int64_t elems = 0;
    if (!mul3(N, K, num_experts, &elems)) return MXFP8_ERR_INVALID_ARG;
    return zero_fill_output(C_dev, elems, out_dtype, stream);
  }
  if (!wgrad && K == 0) return zero_fill_output(C_dev, total_rows * N, out_dtype, stream);
  int st = gemm_checks(A_dev, sA_dev, B_dev, sB_dev, C_dev, op, out_dtype);
  if (st != MXFP8_OK) return st;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != MXFP8_OK) return st;
  GemmArgs a{A_dev, sA_dev, B_dev, sB_dev, C_dev, 0, N, K, op, out_dtype,
             expert_offsets_dev, num_experts, total_rows, d->status};
  return launch_grouped_gemm(a, static_cast<cudaStream_t>(stream));
}

size_t mxfp8_selfcheck_workspace_bytes(int64_t tokens, int64_t N, int64_t K) {
  if (tokens <= 0 || N <= 0 || K <= 0 || K % 32 || N % 16 || tokens % 16) return 0;
  const int64_t b = selfcheck_workspace_bytes(tokens, N, K);
  return b < 0 ? 0 : static_cast<size_t>(b);
}

int mxfp8_selfcheck(const void* w_codes_dev, const void* w_scales_dev,
                    const void* ref_codes_dev, const void* ref_scales_dev, int64_t N, int64_t K,
                    const void* x_bf16_dev, int64_t tokens, void* workspace_dev,
                    size_t workspace_bytes, float* rel_err_dev, void* stream) {
  if (!w_codes_dev || !w_scales_dev || !ref_codes_dev || !ref_scales_dev || !x_bf16_dev ||
      !workspace_dev || !rel_err_dev)
    return MXFP8_ERR_INVALID_ARG;
  if (tokens <= 0 || N <= 0 || K <= 0) return MXFP8_ERR_INVALID_ARG;
  if (K % 32 || N % 16 || tokens % 16) return MXFP8_ERR_ALIGNMENT;
  if (tokens > 0x7FFFFF00 || N > 0x7FFFFF00 || K > 0x7FFFFF00) return MXFP8_ERR_INVALID_ARG;
  if (tokens > kMaxSelfcheckTokens) return MXFP8_ERR_INVALID_ARG;
  const int64_t need = selfcheck_workspace_bytes(tokens, N, K);
  if (need < 0 || workspace_bytes < static_cast<size_t>(need)) return MXFP8_ERR_INVALID_ARG;
  if (!aligned16(w_codes_dev) || !aligned16(w_scales_dev) || !aligned16(x_bf16_dev) ||
      (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) ||
      (reinterpret_cast<uintptr_t>(rel_err_dev) & 3u))
    return MXFP8_ERR_ALIGNMENT;
  DeviceState* d = nullptr;
  const int st = device_state(&d);
  if (st != MXFP8_OK) return st;
  SelfcheckArgs a{w_codes_dev, w_scales_dev, ref_codes_dev, ref_scales_dev, N, K, x_bf16_dev,
                  tokens, workspace_dev, rel_err_dev, d->status};
  return launch_selfcheck(a, static_cast<cudaStream_t>(stream));
}

int mxfp8_selfcheck_noalloc(const void* w_codes_dev, const void* w_scales_dev,
                            const void* ref_codes_dev, const void* ref_scales_dev, int64_t N,
                            int64_t K, const void* x_bf16_dev, int64_t tokens,
                            float* rel_err_dev, void* stream) {
  if (!w_codes_dev || !w_scales_dev || !ref_codes_dev || !ref_scales_dev || !x_bf16_dev ||
      !rel_err_dev)
    return MXFP8_ERR_INVALID_ARG;
  if (tokens <= 0 || N <= 0 || K <= 0) return MXFP8_ERR_INVALID_ARG;
  if (K % 32 || N % 16 || tokens % 16) return MXFP8_ERR_ALIGNMENT;
  if (tokens > 0x7FFFFF00 || N > 0x7FFFFF00 || K > 0x7FFFFF00) return MXFP8_ERR_INVALID_ARG;
  if (tokens > kMaxSelfcheckTokens) return MXFP8_ERR_INVALID_ARG;
  const int64_t need = selfcheck_workspace_bytes(tokens, N, K);
  if (need < 0 || need > kSelfcheckNoallocMaxBytes) return MXFP8_ERR_INVALID_ARG;
  if (!aligned16(w_codes_dev) || !aligned16(w_scales_dev) || !aligned16(x_bf16_dev) ||
      (reinterpret_cast<uintptr_t>(rel_err_dev) & 3u))
    return MXFP8_ERR_ALIGNMENT;
  DeviceState* d = nullptr;
  int st = device_state(&d);
  if (st != MXFP8_OK) return st;
  void* ws = nullptr;
  st = selfcheck_noalloc_workspace(&ws);
  if (st != MXFP8_OK) return st;
  SelfcheckArgs a{w_codes_dev, w_scales_dev, ref_codes_dev, ref_scales_dev, N, K, x_bf16_dev,
                  tokens, ws, rel_err_dev, d->status};
  return launch_selfcheck(a, static_cast<cudaStream_t>(stream));
}

int mxfp8_set_wait_limit_ns(uint64_t ns) {
  set_wait_limit_ns(ns);
  return MXFP8_OK;
}

int mxfp8_get_device_status(void* stream) {
  DeviceState* d = nullptr;
  const int st = device_state(&d);
  if (st != MXFP8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned slot = g_status_slot.fetch_add(1, std::memory_order_relaxed) % kStatusSlots;
  void* args[] = {const_cast<unsigned*>(&slot)};  // enqueued after the stream's earlier work
  if (cudaLaunchKernel(reinterpret_cast<const void*>(take_status_kernel), dim3(1), dim3(1), args,
                       0, s) != cudaSuccess)
    return MXFP8_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_status_taken, sizeof(int), slot * sizeof(int),
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MXFP8_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MXFP8_ERR_CUDA;
  return v;
}

}  // extern "C"

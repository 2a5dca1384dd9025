// internal.h - host-side interface between the C ABI (api.cu) and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxfp8 {

constexpr int kAxisBoth = 2;  // both copies from one read (row-wise + column-wise)

struct QuantizeArgs {
  const void* src;
  int64_t batch;          // independent matrices (1 for a plain call)
  int64_t rows, cols;     // one matrix
  int axis;               // MXFP8_AXIS_ROW / COL, or kAxisBoth
  void* out;              // ROW or COL output (ROW output when axis == kAxisBoth)
  void* scales;
  int64_t scale_item_bytes;
  void* out_col;          // kAxisBoth: the column-wise output
  void* scales_col;
  int64_t scale_item_bytes_col;
  int layout;             // MXFP8_SCALES_LINEAR / SWIZZLED
  const int32_t* offsets; // grouped call: device [num_experts + 1], else nullptr
  int num_experts;
  int rule;               // MXFP8_RULE_FLOOR / MXFP8_RULE_CEIL
  int* status;            // device status word
};

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t stream);

// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialization (its kernels wait for the previous kernel of the
// stream in the kernel itself), unless the environment sets MXFP8_PDL=0 (read once).
// Writes the launch attribute to *attr and returns 1, or returns 0 when it is off.
int pdl_attr(cudaLaunchAttribute* attr);

// Several dual (row-wise + column-wise) quantizations in one launch.
constexpr int kMaxQuantizeJobs = 8;
struct QuantizeJobs {
  int n;
  int layout;
  const void* src[kMaxQuantizeJobs];
  int64_t rows[kMaxQuantizeJobs], cols[kMaxQuantizeJobs];
  void* out[kMaxQuantizeJobs];
  void* scales[kMaxQuantizeJobs];
  void* out_col[kMaxQuantizeJobs];
  void* scales_col[kMaxQuantizeJobs];
  int* status;
};

cudaError_t launch_quantize_jobs(const QuantizeJobs& j, cudaStream_t stream);

// FP8 block-wise (128 x 128) weight quantization; scale_inv [ceil(rows/128)][ceil(cols/128)].
cudaError_t launch_blockwise(const void* src, int64_t rows, int64_t cols, void* out,
                             float* scale_inv, bool pow2, cudaStream_t stream);

struct GemmArgs {
  const void* A;
  const void* sA;
  const void* B;
  const void* sB;
  void* C;
  int64_t M, N, K;
  int op;
  int out_dtype;
  // grouped call
  const int32_t* offsets;  // nullptr for the dense GEMM
  int num_experts;
  int64_t total_rows;
  int* status;
  // dense call: caller-owned workspace for a split-K last wave (nullptr: none)
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
};

// Returns MXFP8_OK or an mxfp8_status code.
int launch_gemm(const GemmArgs& a, cudaStream_t stream);
// Bytes of workspace with which launch_gemm runs this dense GEMM's last wave as split-K
// pieces on the current device (0: it never does).
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int out_dtype);
int launch_grouped_gemm(const GemmArgs& a, cudaStream_t stream);

struct SelfcheckArgs {
  const void* w_codes;   // E4M3 [N][K] as the GEMM reads it
  const void* w_scales;  // swizzled scales as the GEMM reads them
  const void* ref_codes;   // canonical synchronized weight, E4M3 [N][K]
  const void* ref_scales;  // its linear scales [N][K/32]
  int64_t N, K;
  const void* x;         // BF16 [T][K]
  int64_t T;
  void* workspace;       // selfcheck_workspace_bytes(T, N, K) bytes
  float* rel_err;        // device, one float
  int* status;
};

int64_t selfcheck_workspace_bytes(int64_t T, int64_t N, int64_t K);

// Size of the fixed workspace behind mxfp8_selfcheck_noalloc (8 MiB).
constexpr int64_t kSelfcheckNoallocMaxBytes = int64_t(8) << 20;
int selfcheck_noalloc_workspace(void** out);
int launch_selfcheck(const SelfcheckArgs& a, cudaStream_t stream);

int num_sms();  // of the current device (cached)

// Pipeline wait limit of the GEMM kernels for later launches (0: the default).
void set_wait_limit_ns(uint64_t ns);

}  // namespace mxfp8

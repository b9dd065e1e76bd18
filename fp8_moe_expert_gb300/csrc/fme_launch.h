// fme_launch.h -- host-side launch descriptions passed from the C ABI layer
// (api.cu, which validates arguments) to the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fme {

struct LaunchNvfp4 {
  const void *x;
  int64_t rows, k;
  const int32_t *offsets;
  int32_t num_groups;
  uint8_t *codes, *sf;
  float *row_scale;
  int32_t *status;
  int num_sms;
  cudaStream_t stream;
  bool swiglu = false;         // x is a gate/up output [rows x 2k]; quantize silu(gate) * up
  void *h_out = nullptr;       // swiglu: the bf16 activation [rows x k], or NULL
  const int32_t *gather = nullptr;  // row r reads input row gather[r] / gather_div (permuted tokens)
  int32_t gather_div = 1;
  int64_t gather_limit = 0;         // input rows; gathered rows outside [0, limit) are reported
  const float *tensor_amax = nullptr;  // standard NVFP4: every row scaled by this amax (device)
};

struct LaunchRoute {
  const int32_t *ids;
  int64_t tokens;
  int32_t top_k, num_experts;
  int32_t *offsets, *row_of, *src_row;
  int32_t *ws;  // [chunks x num_experts]
  int32_t *status;
  cudaStream_t stream;
};

struct LaunchCombine {
  const void *y;
  const int32_t *row_of;
  const float *weights;
  int64_t tokens;
  int32_t top_k;
  int64_t n, rows_y;
  void *out;
  int32_t *status;
  int num_sms;
  cudaStream_t stream;
};

struct LaunchMxfp8 {
  const void *x;
  int64_t rows, cols;
  const int32_t *offsets;
  int32_t num_groups;
  uint8_t *codes, *sf;
  int32_t *padded_offsets;  // column-wise only
  int64_t ld;               // column-wise only
  int32_t *status;
  int num_sms;
  cudaStream_t stream;
  // Row-wise only: row r reads source row gather[r] / gather_div, which must lie
  // in [0, gather_limit).
  const int32_t *gather = nullptr;
  int32_t gather_div = 1;
  int64_t gather_limit = 0;
  // SwiGLU backward (launch_swiglu_bwd_mxfp8): x = gate/up [rows x cols], dh
  // [rows x cols/2], optional bf16 d(gate/up) out [rows x cols].
  const void *dh = nullptr;
  void *d_out = nullptr;
  bool ceil_scale = false;  // row-wise / column-wise only: X = 2^ceil(log2(amax / 448))
};

// kFwdNvfp4Swiglu: the NVFP4 forward of the gate/up projection with h = silu(gate) * up
// formed in the epilogue (output [rows x n / 2]).
enum class GemmKind { kFwdNvfp4 = 0, kDgradMxfp8 = 1, kWgradMxfp8 = 2, kFwdMxfp8 = 3, kFwdNvfp4Swiglu = 4 };
__host__ __device__ constexpr bool is_fwd_nvfp4(GemmKind k) {
  return k == GemmKind::kFwdNvfp4 || k == GemmKind::kFwdNvfp4Swiglu;
}

struct LaunchGemm {
  GemmKind kind;
  CUtensorMap map_a, map_b;      // operand codes, uint8, 128-byte swizzle
  CUtensorMap map_sfa, map_sfb;  // tiled scales viewed as [128-row blocks x 8-byte words]
  CUtensorMap map_y;             // the bf16 output [rows x n], 32 x 32 boxes, 64-byte swizzle (not the fp32 accumulate)
  const float *a_scale, *b_scale;  // forward only
  const int32_t *offsets;          // row offsets (fwd, dgrad) or padded offsets (wgrad)
  int32_t num_experts;
  int64_t m, n, k;          // GEMM sizes; k unused for wgrad (per-expert)
  int64_t lda, ldb;         // wgrad: position extents of A and B; dgrad: ldb
  void *y;
  int32_t *status;
  int num_sms;
  int stages;  // operand ring depth, set by launch_grouped_gemm
  cudaStream_t stream;
  bool accumulate = false;  // wgrad only: y is fp32 and receives y += result
};

cudaError_t launch_quantize_nvfp4(const LaunchNvfp4 &a);
// Standard NVFP4 (one FP32 scale for the whole tensor): zero *tensor_amax, reduce
// max |x| into it, then quantize every row with it in place of the row's amax.
cudaError_t launch_quantize_nvfp4_pertensor(const LaunchNvfp4 &a, float *tensor_amax);
cudaError_t launch_quantize_mxfp8_rows(const LaunchMxfp8 &a);
cudaError_t launch_quantize_mxfp8_cols(const LaunchMxfp8 &a);
cudaError_t launch_quantize_mxfp8_rowcol(const LaunchMxfp8 &a, uint8_t *row_codes, uint8_t *row_sf);
// Fused SwiGLU backward + row-wise and column-wise MXFP8 of d(gate/up); a.codes /
// a.sf are the column-wise outputs (as launch_quantize_mxfp8_rowcol).
cudaError_t launch_swiglu_bwd_mxfp8(const LaunchMxfp8 &a, uint8_t *row_codes, uint8_t *row_sf);
cudaError_t launch_grouped_gemm(const LaunchGemm &a);
cudaError_t launch_route(const LaunchRoute &r);
// launch_route with the module's static device counters as the workspace (r.ws
// is ignored); needs chunks * num_experts <= kRouteStaticWords.
constexpr int64_t kRouteStaticWords = int64_t(1) << 20;
cudaError_t launch_route_static(LaunchRoute r);
cudaError_t launch_combine(const LaunchCombine &c);
constexpr int64_t kRouteChunkHost = 1024;  // assignments per routing chunk (route.cu)

}  // namespace fme

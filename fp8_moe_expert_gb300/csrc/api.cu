// api.cu -- the extern "C" boundary of libfme.so (declared in include/fme.h):
// host-side argument checks, device checks, TMA descriptor encoding, launches.
// Nothing here allocates device memory or synchronises a stream, except
// fme_read_device_status, which is documented to synchronise.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/fme.h"
#include "fme_launch.h"

namespace {

thread_local std::string g_last_cuda_error;

fme_status cuda_fail(cudaError_t err, const char *where) {
  g_last_cuda_error = std::string(where) + ": " + cudaGetErrorString(err);
  return FME_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device facts, looked up once per device.
struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 supported, 2 unsupported
  int num_sms = 0;
};
DeviceInfo g_devices[64];
std::mutex g_device_mutex;

fme_status current_device(int *num_sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return FME_ERR_UNSUPPORTED_DEVICE;
  DeviceInfo &d = g_devices[dev];
  if (d.state.load(std::memory_order_acquire) == 0) {
    std::lock_guard<std::mutex> lock(g_device_mutex);
    if (d.state.load(std::memory_order_relaxed) == 0) {
      int major = 0, minor = 0, sms = 0;
      if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
          (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
          (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(err, "cudaDeviceGetAttribute");
      d.num_sms = sms;
      d.state.store((major == 10 && minor == 3) ? 1 : 2, std::memory_order_release);
    }
  }
  if (d.state.load(std::memory_order_acquire) != 1) return FME_ERR_UNSUPPORTED_DEVICE;
  *num_sms = d.num_sms;
  return FME_OK;
}

// cuTensorMapEncodeTiled from the driver, fetched once through the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

fme_status get_encoder(EncodeTiledFn *fn) {
  std::call_once(g_encode_once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (g_encode == nullptr) {
    g_last_cuda_error = "cuTensorMapEncodeTiled not available from the driver";
    return FME_ERR_CUDA;
  }
  *fn = g_encode;
  return FME_OK;
}

// 2-D uint8 tensor [rows x inner] (row stride `stride` bytes), box {128 bytes, box_rows},
// 128-byte swizzle, zero fill out of bounds.
fme_status encode_u8_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint64_t stride,
                        uint32_t box_rows) {
  EncodeTiledFn fn;
  fme_status st = get_encoder(&fn);
  if (st != FME_OK) return st;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {stride};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    g_last_cuda_error = buf;
    return FME_ERR_CUDA;
  }
  return FME_OK;
}

// bf16 matrix [rows x cols] (row stride cols * 2 bytes) for bulk tensor stores of
// 32 x 32 boxes with the 64-byte swizzle.
fme_status encode_bf16_out(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn;
  fme_status st = get_encoder(&fn);
  if (st != FME_OK) return st;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (output) failed (CUresult %d)", static_cast<int>(r));
    g_last_cuda_error = buf;
    return FME_ERR_CUDA;
  }
  return FME_OK;
}

// Tiled scales of a tensor as a 2-D map of 8-byte words: one row per 128-row
// block (`row_bytes` bytes each), boxes of `box_tiles` 512-byte tiles x `box_rows`
// blocks, no swizzle, zero fill out of bounds.
fme_status encode_scales_2d(CUtensorMap *map, const void *base, uint64_t row_blocks, uint64_t row_bytes,
                            uint32_t box_tiles, uint32_t box_rows) {
  EncodeTiledFn fn;
  fme_status st = get_encoder(&fn);
  if (st != FME_OK) return st;
  cuuint64_t dims[2] = {row_bytes / 8, row_blocks};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {64 * box_tiles, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (scales) failed (CUresult %d)", static_cast<int>(r));
    g_last_cuda_error = buf;
    return FME_ERR_CUDA;
  }
  return FME_OK;
}

int64_t padded_rows_bound(int64_t rows, int32_t groups) {
  if (rows < 0 || groups < 1) return 0;
  return ((rows + 127 * static_cast<int64_t>(groups)) / 128) * 128;
}

fme_status check_groups(int32_t num_groups) {
  return (num_groups < 1 || num_groups > FME_MAX_GROUPS) ? FME_ERR_INVALID_ARGUMENT : FME_OK;
}

}  // namespace

extern "C" {

int64_t fme_sf_padded_rows(int64_t rows, int32_t num_groups) { return padded_rows_bound(rows, num_groups); }

int64_t fme_sf_bytes(int64_t rows, int64_t cols, int32_t block, int32_t num_groups) {
  if (cols < 0 || block <= 0 || cols % block) return 0;
  const int64_t c4 = ((cols / block) + 3) / 4 * 4;
  return padded_rows_bound(rows, num_groups) * c4;
}

int64_t fme_colwise_ld(int64_t rows, int32_t num_groups) { return padded_rows_bound(rows, num_groups); }

int64_t fme_route_workspace_bytes(int64_t tokens, int32_t top_k, int32_t num_experts) {
  if (tokens < 0 || top_k < 1 || num_experts < 1) return 0;
  const int64_t chunks = (tokens * top_k + fme::kRouteChunkHost - 1) / fme::kRouteChunkHost;
  const int64_t b = chunks * num_experts * 4;
  return b < 16 ? 16 : b;
}

const char *fme_version(void) { return "fme 0.1.0 (sm_103a)"; }

const char *fme_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

const char *fme_error_string(fme_status status) {
  switch (status) {
    case FME_OK: return "ok";
    case FME_ERR_INVALID_ARGUMENT: return "invalid argument";
    case FME_ERR_MISALIGNED: return "pointer or leading dimension not 16-byte aligned";
    case FME_ERR_UNSUPPORTED_SHAPE: return "shape outside the supported tiling";
    case FME_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (GB300)";
    case FME_ERR_CUDA: return "CUDA error";
    case FME_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
    case FME_ERR_DEVICE_BAD_OFFSETS: return "offsets do not rise from 0 to rows";
    case FME_ERR_DEVICE_BAD_INDEX: return "an expert id or a row index out of range";
    default: return "unknown status";
  }
}

fme_status fme_read_device_status(const int32_t *dev_status, void *stream, int32_t *raw) {
  if (dev_status == nullptr) return FME_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  cudaError_t err = cudaMemcpyAsync(&host, dev_status, sizeof host, cudaMemcpyDeviceToHost, s);
  if (err != cudaSuccess) return cuda_fail(err, "cudaMemcpyAsync(status)");
  err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return cuda_fail(err, "cudaStreamSynchronize");
  if (raw) *raw = host;
  if (host & FME_DEV_BAD_OFFSETS) return FME_ERR_DEVICE_BAD_OFFSETS;
  if (host & FME_DEV_BAD_INDEX) return FME_ERR_DEVICE_BAD_INDEX;
  if (host & FME_DEV_TIMEOUT) return FME_ERR_DEVICE_TIMEOUT;
  return FME_OK;
}

fme_status quantize_nvfp4_pertoken(const void *x, int64_t rows, int64_t k, const int32_t *offsets,
                                   int32_t num_groups, uint8_t *codes, uint8_t *sf, float *row_scale,
                                   int32_t *dev_status, void *stream) {
  if (rows < 0 || check_groups(num_groups) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (offsets == nullptr && num_groups != 1) return FME_ERR_INVALID_ARGUMENT;
  if (k % 64 != 0 || k < 64 || k > 8192) return FME_ERR_UNSUPPORTED_SHAPE;
  if (rows > (int64_t(1) << 31) - 1) return FME_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return FME_OK;
  if (!x || !codes || !sf || !row_scale) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf) || !aligned16(row_scale)) return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchNvfp4 a{x, rows, k, offsets, num_groups, codes, sf, row_scale, dev_status, sms,
                     static_cast<cudaStream_t>(stream)};
  cudaError_t err = fme::launch_quantize_nvfp4(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "quantize_nvfp4_pertoken launch");
}

fme_status quantize_nvfp4_pertensor(const void *x, int64_t rows, int64_t k, const int32_t *offsets,
                                    int32_t num_groups, uint8_t *codes, uint8_t *sf, float *row_scale,
                                    float *tensor_amax, int32_t *dev_status, void *stream) {
  if (rows < 0 || check_groups(num_groups) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (offsets == nullptr && num_groups != 1) return FME_ERR_INVALID_ARGUMENT;
  if (k % 64 != 0 || k < 64 || k > 8192) return FME_ERR_UNSUPPORTED_SHAPE;
  if (rows > (int64_t(1) << 31) - 1 - 128 * static_cast<int64_t>(num_groups)) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!tensor_amax) return FME_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!x || !codes || !sf || !row_scale)) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf) || !aligned16(row_scale) || !aligned16(tensor_amax))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchNvfp4 a{x, rows, k, offsets, num_groups, codes, sf, row_scale, dev_status, sms,
                     static_cast<cudaStream_t>(stream)};
  cudaError_t err = fme::launch_quantize_nvfp4_pertensor(a, tensor_amax);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "quantize_nvfp4_pertensor launch");
}

fme_status swiglu_quantize_nvfp4(const void *gate_up, int64_t rows, int64_t inter, const int32_t *offsets,
                                 int32_t num_groups, uint8_t *codes, uint8_t *sf, float *row_scale, void *h,
                                 int32_t *dev_status, void *stream) {
  if (rows < 0 || check_groups(num_groups) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (offsets == nullptr && num_groups != 1) return FME_ERR_INVALID_ARGUMENT;
  if (inter % 64 != 0 || inter < 64 || inter > 8192) return FME_ERR_UNSUPPORTED_SHAPE;
  if (rows > (int64_t(1) << 31) - 1) return FME_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return FME_OK;
  if (!gate_up || !codes || !sf || !row_scale) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(gate_up) || !aligned16(codes) || !aligned16(sf) || !aligned16(row_scale) || !aligned16(h))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchNvfp4 a{gate_up, rows, inter, offsets, num_groups, codes, sf, row_scale, dev_status, sms,
                     static_cast<cudaStream_t>(stream)};
  a.swiglu = true;
  a.h_out = h;
  cudaError_t err = fme::launch_quantize_nvfp4(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "swiglu_quantize_nvfp4 launch");
}

fme_status moe_route(const int32_t *topk_ids, int64_t tokens, int32_t top_k, int32_t num_experts, int32_t *offsets,
                     int32_t *row_of, int32_t *src_row, void *workspace, int64_t workspace_bytes,
                     int32_t *dev_status, void *stream) {
  if (tokens < 0 || top_k < 1 || top_k > 64 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (tokens * top_k > (int64_t(1) << 31) - 1) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!offsets || !workspace) return FME_ERR_INVALID_ARGUMENT;
  if (tokens > 0 && (!topk_ids || !row_of || !src_row)) return FME_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < fme_route_workspace_bytes(tokens, top_k, num_experts)) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(topk_ids) || !aligned16(offsets) || !aligned16(row_of) || !aligned16(src_row) ||
      !aligned16(workspace))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchRoute r{topk_ids, tokens, top_k, num_experts, offsets, row_of, src_row,
                     static_cast<int32_t *>(workspace), dev_status, static_cast<cudaStream_t>(stream)};
  cudaError_t err = fme::launch_route(r);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "moe_route launch");
}

fme_status moe_route_noalloc(const int32_t *topk_ids, int64_t tokens, int32_t top_k, int32_t num_experts,
                             int32_t *offsets, int32_t *row_of, int32_t *src_row, int32_t *dev_status,
                             void *stream) {
  if (tokens < 0 || top_k < 1 || top_k > 64 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (tokens * top_k > (int64_t(1) << 31) - 1) return FME_ERR_UNSUPPORTED_SHAPE;
  const int64_t chunks = (tokens * top_k + fme::kRouteChunkHost - 1) / fme::kRouteChunkHost;
  if (chunks * num_experts > fme::kRouteStaticWords) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!offsets) return FME_ERR_INVALID_ARGUMENT;
  if (tokens > 0 && (!topk_ids || !row_of || !src_row)) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(topk_ids) || !aligned16(offsets) || !aligned16(row_of) || !aligned16(src_row))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchRoute r{topk_ids, tokens, top_k, num_experts, offsets, row_of, src_row, nullptr, dev_status,
                     static_cast<cudaStream_t>(stream)};
  cudaError_t err = fme::launch_route_static(r);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "moe_route_noalloc launch");
}

fme_status permute_quantize_nvfp4(const void *x, int64_t tokens, int64_t k, const int32_t *src_row, int32_t top_k,
                                  const int32_t *offsets, int32_t num_experts, uint8_t *codes, uint8_t *sf,
                                  float *row_scale, int32_t *dev_status, void *stream) {
  if (tokens < 0 || top_k < 1 || top_k > 64 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (k % 64 != 0 || k < 64 || k > 8192) return FME_ERR_UNSUPPORTED_SHAPE;
  const int64_t rows = tokens * top_k;
  if (rows > (int64_t(1) << 31) - 1) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!offsets) return FME_ERR_INVALID_ARGUMENT;
  if (rows == 0) return FME_OK;
  if (!x || !src_row || !codes || !sf || !row_scale) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(src_row) || !aligned16(codes) || !aligned16(sf) || !aligned16(row_scale) ||
      !aligned16(offsets))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchNvfp4 a{x, rows, k, offsets, num_experts, codes, sf, row_scale, dev_status, sms,
                     static_cast<cudaStream_t>(stream)};
  a.gather = src_row;
  a.gather_div = top_k;
  a.gather_limit = tokens;
  cudaError_t err = fme::launch_quantize_nvfp4(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "permute_quantize_nvfp4 launch");
}

fme_status permute_quantize_mxfp8(const void *x, int64_t tokens, int64_t k, const int32_t *src_row, int32_t top_k,
                                  const int32_t *offsets, int32_t num_experts, uint8_t *codes, uint8_t *sf,
                                  int32_t *dev_status, void *stream) {
  if (tokens < 0 || top_k < 1 || top_k > 64 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (k % 32 != 0 || k < 32 || k > 65536) return FME_ERR_UNSUPPORTED_SHAPE;
  const int64_t rows = tokens * top_k;
  if (rows > (int64_t(1) << 31) - 1 - 128 * static_cast<int64_t>(num_experts)) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!offsets) return FME_ERR_INVALID_ARGUMENT;
  if (rows == 0) return FME_OK;
  if (!x || !src_row || !codes || !sf) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(src_row) || !aligned16(codes) || !aligned16(sf)) return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchMxfp8 a{x, rows, k, offsets, num_experts, codes, sf, nullptr, 0, dev_status, sms,
                     static_cast<cudaStream_t>(stream)};
  a.gather = src_row;
  a.gather_div = top_k;
  a.gather_limit = tokens;
  cudaError_t err = fme::launch_quantize_mxfp8_rows(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "permute_quantize_mxfp8 launch");
}

fme_status moe_combine(const void *y, int64_t rows_y, const int32_t *row_of, const float *weights, int64_t tokens,
                       int32_t top_k, int64_t n, void *out, int32_t *dev_status, void *stream) {
  if (tokens < 0 || rows_y < 0 || top_k < 1 || top_k > 64 || n < 0) return FME_ERR_INVALID_ARGUMENT;
  if (n % 8 != 0 || n == 0) return FME_ERR_UNSUPPORTED_SHAPE;
  if (tokens * top_k > (int64_t(1) << 31) - 1) return FME_ERR_UNSUPPORTED_SHAPE;
  if (tokens == 0) return FME_OK;
  if (!row_of || !weights || !out || (rows_y > 0 && !y)) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(y) || !aligned16(row_of) || !aligned16(weights) || !aligned16(out)) return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchCombine c{y, row_of, weights, tokens, top_k, n, rows_y, out, dev_status, sms,
                       static_cast<cudaStream_t>(stream)};
  cudaError_t err = fme::launch_combine(c);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "moe_combine launch");
}

fme_status quantize_mxfp8(const void *x, int64_t rows, int64_t cols, int32_t axis, const int32_t *offsets,
                          int32_t num_groups, uint8_t *codes, uint8_t *sf, int32_t *padded_offsets,
                          int32_t *dev_status, void *stream) {
  const bool ceil_scale = (axis & FME_MX_SCALE_CEIL) != 0;
  axis &= ~FME_MX_SCALE_CEIL;
  if (rows < 0 || check_groups(num_groups) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (offsets == nullptr && num_groups != 1) return FME_ERR_INVALID_ARGUMENT;
  if (axis != FME_ROWWISE && axis != FME_COLWISE) return FME_ERR_INVALID_ARGUMENT;
  if (rows > (int64_t(1) << 31) - 1 - 128 * static_cast<int64_t>(num_groups)) return FME_ERR_UNSUPPORTED_SHAPE;
  if (axis == FME_ROWWISE) {
    if (padded_offsets != nullptr) return FME_ERR_INVALID_ARGUMENT;
    if (cols % 32 != 0 || cols < 32 || cols > 65536) return FME_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return FME_OK;
  } else {
    if (cols % 128 != 0 || cols < 128 || cols > 65536) return FME_ERR_UNSUPPORTED_SHAPE;
    if (padded_offsets == nullptr) return FME_ERR_INVALID_ARGUMENT;
    if (!aligned16(padded_offsets)) return FME_ERR_MISALIGNED;
  }
  if ((!x && rows > 0) || !codes || !sf) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf)) return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchMxfp8 a{x, rows, cols, offsets, num_groups, codes, sf, padded_offsets,
                     fme_colwise_ld(rows, num_groups), dev_status, sms, static_cast<cudaStream_t>(stream)};
  a.ceil_scale = ceil_scale;
  cudaError_t err =
      (axis == FME_ROWWISE) ? fme::launch_quantize_mxfp8_rows(a) : fme::launch_quantize_mxfp8_cols(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "quantize_mxfp8 launch");
}

fme_status quantize_mxfp8_rowcol(const void *x, int64_t rows, int64_t cols, const int32_t *offsets,
                                 int32_t num_groups, uint8_t *row_codes, uint8_t *row_sf, uint8_t *col_codes,
                                 uint8_t *col_sf, int32_t *padded_offsets, int32_t *dev_status, void *stream) {
  if (rows < 0 || check_groups(num_groups) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (offsets == nullptr && num_groups != 1) return FME_ERR_INVALID_ARGUMENT;
  if (rows > (int64_t(1) << 31) - 1 - 128 * static_cast<int64_t>(num_groups)) return FME_ERR_UNSUPPORTED_SHAPE;
  if (cols % 128 != 0 || cols < 128 || cols > 65536) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!padded_offsets || !col_codes || !col_sf || !row_sf || (rows > 0 && (!x || !row_codes)))
    return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(row_codes) || !aligned16(row_sf) || !aligned16(col_codes) || !aligned16(col_sf) ||
      !aligned16(padded_offsets))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchMxfp8 a{x, rows, cols, offsets, num_groups, col_codes, col_sf, padded_offsets,
                     fme_colwise_ld(rows, num_groups), dev_status, sms, static_cast<cudaStream_t>(stream)};
  cudaError_t err = fme::launch_quantize_mxfp8_rowcol(a, row_codes, row_sf);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "quantize_mxfp8_rowcol launch");
}

fme_status swiglu_backward_quantize_mxfp8(const void *gate_up, const void *dh, int64_t rows, int64_t inter,
                                          const int32_t *offsets, int32_t num_groups, uint8_t *row_codes,
                                          uint8_t *row_sf, uint8_t *col_codes, uint8_t *col_sf,
                                          int32_t *padded_offsets, void *d_gate_up, int32_t *dev_status,
                                          void *stream) {
  if (rows < 0 || check_groups(num_groups) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (offsets == nullptr && num_groups != 1) return FME_ERR_INVALID_ARGUMENT;
  if (rows > (int64_t(1) << 31) - 1 - 128 * static_cast<int64_t>(num_groups)) return FME_ERR_UNSUPPORTED_SHAPE;
  if (inter % 128 != 0 || inter < 128 || inter > 32768) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!padded_offsets || !col_codes || !col_sf || !row_sf || (rows > 0 && (!gate_up || !dh || !row_codes)))
    return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(gate_up) || !aligned16(dh) || !aligned16(row_codes) || !aligned16(row_sf) ||
      !aligned16(col_codes) || !aligned16(col_sf) || !aligned16(padded_offsets) || !aligned16(d_gate_up))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchMxfp8 a{gate_up, rows, 2 * inter, offsets, num_groups, col_codes, col_sf, padded_offsets,
                     fme_colwise_ld(rows, num_groups), dev_status, sms, static_cast<cudaStream_t>(stream)};
  a.dh = dh;
  a.d_out = d_gate_up;
  cudaError_t err = fme::launch_swiglu_bwd_mxfp8(a, row_codes, row_sf);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "swiglu_backward_quantize_mxfp8 launch");
}

// The NVFP4 forward, plain (y [m x n]) or with the SwiGLU epilogue (y = h [m x n / 2]).
static fme_status fwd_nvfp4(bool swiglu, const uint8_t *a_codes, const uint8_t *a_sf, const float *a_scale,
                            const uint8_t *b_codes, const uint8_t *b_sf, const float *b_scale, const int32_t *offsets,
                            int32_t num_experts, int64_t m, int64_t n, int64_t k, void *y, int32_t *dev_status,
                            void *stream) {
  if (m < 0 || n < 0 || k < 0 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (n % 256 != 0 || n == 0 || k % 256 != 0 || k == 0 || k > 65536) return FME_ERR_UNSUPPORTED_SHAPE;
  if (m > (int64_t(1) << 31) - 1 || static_cast<int64_t>(num_experts) * n > (int64_t(1) << 31) - 1)
    return FME_ERR_UNSUPPORTED_SHAPE;
  if (!offsets) return FME_ERR_INVALID_ARGUMENT;
  if (m == 0) return FME_OK;
  if (!a_codes || !a_sf || !a_scale || !b_codes || !b_sf || !b_scale || !y) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(a_codes) || !aligned16(a_sf) || !aligned16(a_scale) || !aligned16(b_codes) ||
      !aligned16(b_sf) || !aligned16(b_scale) || !aligned16(y) || !aligned16(offsets))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchGemm a{};
  a.kind = swiglu ? fme::GemmKind::kFwdNvfp4Swiglu : fme::GemmKind::kFwdNvfp4;
  if ((st = encode_u8_2d(&a.map_a, a_codes, k / 2, m, k / 2, 128)) != FME_OK) return st;
  if ((st = encode_u8_2d(&a.map_b, b_codes, k / 2, static_cast<uint64_t>(num_experts) * n, k / 2, 128)) != FME_OK)
    return st;
  // scales: (k / 64) tiles of 512 bytes per 128-row block; a stage takes 4 tiles
  if ((st = encode_scales_2d(&a.map_sfa, a_sf, padded_rows_bound(m, num_experts) / 128, (k / 64) * 512, 4, 1)) !=
      FME_OK)
    return st;
  // B scales: the same tiled layout (the stacked weights are one group of
  // num_experts * n rows); a stage takes 4 tiles of each of the tile's two 128-row
  // blocks, adjacent (one copy) or, with SwiGLU, a gate and an up block (two copies)
  if ((st = encode_scales_2d(&a.map_sfb, b_sf, static_cast<uint64_t>(num_experts) * n / 128, (k / 64) * 512, 4,
                             swiglu ? 1 : 2)) != FME_OK)
    return st;
  if ((st = encode_bf16_out(&a.map_y, y, swiglu ? n / 2 : n, m)) != FME_OK) return st;
  a.a_scale = a_scale;
  a.b_scale = b_scale;
  a.offsets = offsets;
  a.num_experts = num_experts;
  a.m = m;
  a.n = n;
  a.k = k;
  a.y = y;
  a.status = dev_status;
  a.num_sms = sms;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t err = fme::launch_grouped_gemm(a);
  return err == cudaSuccess ? FME_OK
                            : cuda_fail(err, swiglu ? "grouped_gemm_fwd_nvfp4_swiglu launch" : "grouped_gemm_fwd_nvfp4 launch");
}

fme_status grouped_gemm_fwd_nvfp4(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_scale,
                                  const uint8_t *b_codes, const uint8_t *b_sf, const float *b_scale,
                                  const int32_t *offsets, int32_t num_experts, int64_t m, int64_t n, int64_t k,
                                  void *y, int32_t *dev_status, void *stream) {
  return fwd_nvfp4(false, a_codes, a_sf, a_scale, b_codes, b_sf, b_scale, offsets, num_experts, m, n, k, y,
                   dev_status, stream);
}

fme_status grouped_gemm_fwd_nvfp4_swiglu(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_scale,
                                         const uint8_t *b_codes, const uint8_t *b_sf, const float *b_scale,
                                         const int32_t *offsets, int32_t num_experts, int64_t m, int64_t n,
                                         int64_t k, void *h, int32_t *dev_status, void *stream) {
  return fwd_nvfp4(true, a_codes, a_sf, a_scale, b_codes, b_sf, b_scale, offsets, num_experts, m, n, k, h,
                   dev_status, stream);
}

fme_status grouped_gemm_fwd_mxfp8(const uint8_t *a_codes, const uint8_t *a_sf, const uint8_t *b_codes,
                                  const uint8_t *b_sf, const int32_t *offsets, int32_t num_experts, int64_t m,
                                  int64_t n, int64_t k, void *y, int32_t *dev_status, void *stream) {
  if (m < 0 || n < 0 || k < 0 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (n % 256 != 0 || n == 0 || k % 128 != 0 || k == 0 || k > 65536) return FME_ERR_UNSUPPORTED_SHAPE;
  if (m > (int64_t(1) << 31) - 1 || static_cast<int64_t>(num_experts) * n > (int64_t(1) << 31) - 1)
    return FME_ERR_UNSUPPORTED_SHAPE;
  if (!offsets) return FME_ERR_INVALID_ARGUMENT;
  if (m == 0) return FME_OK;
  if (!a_codes || !a_sf || !b_codes || !b_sf || !y) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(a_codes) || !aligned16(a_sf) || !aligned16(b_codes) || !aligned16(b_sf) || !aligned16(y) ||
      !aligned16(offsets))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchGemm a{};
  a.kind = fme::GemmKind::kFwdMxfp8;
  if ((st = encode_u8_2d(&a.map_a, a_codes, k, m, k, 128)) != FME_OK) return st;
  if ((st = encode_u8_2d(&a.map_b, b_codes, k, static_cast<uint64_t>(num_experts) * n, k, 128)) != FME_OK)
    return st;
  // row-wise E8M0 scales: (k / 128) tiles of 512 bytes per 128-row block; a stage takes one
  if ((st = encode_scales_2d(&a.map_sfa, a_sf, padded_rows_bound(m, num_experts) / 128, (k / 128) * 512, 1, 1)) !=
      FME_OK)
    return st;
  if ((st = encode_scales_2d(&a.map_sfb, b_sf, static_cast<uint64_t>(num_experts) * n / 128, (k / 128) * 512, 1,
                             2)) != FME_OK)
    return st;
  if ((st = encode_bf16_out(&a.map_y, y, n, m)) != FME_OK) return st;
  a.offsets = offsets;
  a.num_experts = num_experts;
  a.m = m;
  a.n = n;
  a.k = k;
  a.y = y;
  a.status = dev_status;
  a.num_sms = sms;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t err = fme::launch_grouped_gemm(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "grouped_gemm_fwd_mxfp8 launch");
}

fme_status grouped_gemm_dgrad_mxfp8(const uint8_t *a_codes, const uint8_t *a_sf, const uint8_t *b_codes,
                                    const uint8_t *b_sf, int64_t ldb, const int32_t *offsets, int32_t num_experts,
                                    int64_t m, int64_t n, int64_t k, void *y, int32_t *dev_status, void *stream) {
  if (m < 0 || n < 0 || k < 0 || ldb < 0 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (n % 256 != 0 || n == 0 || k % 128 != 0 || k == 0 || ldb % 128 != 0) return FME_ERR_UNSUPPORTED_SHAPE;
  if (ldb < static_cast<int64_t>(num_experts) * k) return FME_ERR_INVALID_ARGUMENT;
  if (m > (int64_t(1) << 31) - 1 || ldb > (int64_t(1) << 31) - 1 || k > 65536) return FME_ERR_UNSUPPORTED_SHAPE;
  if (!offsets) return FME_ERR_INVALID_ARGUMENT;
  if (m == 0) return FME_OK;
  if (!a_codes || !a_sf || !b_codes || !b_sf || !y) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(a_codes) || !aligned16(a_sf) || !aligned16(b_codes) || !aligned16(b_sf) || !aligned16(y) ||
      !aligned16(offsets))
    return FME_ERR_MISALIGNED;
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchGemm a{};
  a.kind = fme::GemmKind::kDgradMxfp8;
  if ((st = encode_u8_2d(&a.map_a, a_codes, k, m, k, 128)) != FME_OK) return st;
  if ((st = encode_u8_2d(&a.map_b, b_codes, ldb, n, ldb, 128)) != FME_OK) return st;
  if ((st = encode_scales_2d(&a.map_sfa, a_sf, padded_rows_bound(m, num_experts) / 128, (k / 128) * 512, 1, 1)) !=
      FME_OK)
    return st;
  if ((st = encode_scales_2d(&a.map_sfb, b_sf, n / 128, (ldb / 128) * 512, 1, 2)) != FME_OK) return st;
  if ((st = encode_bf16_out(&a.map_y, y, n, m)) != FME_OK) return st;
  a.offsets = offsets;
  a.num_experts = num_experts;
  a.m = m;
  a.n = n;
  a.k = k;
  a.ldb = ldb;
  a.y = y;
  a.status = dev_status;
  a.num_sms = sms;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t err = fme::launch_grouped_gemm(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, "grouped_gemm_dgrad_mxfp8 launch");
}

static fme_status wgrad_call(const uint8_t *a_codes, const uint8_t *a_sf, int64_t lda, const uint8_t *b_codes,
                             const uint8_t *b_sf, int64_t ldb, const int32_t *padded_offsets, int32_t num_experts,
                             int64_t m, int64_t n, void *y, bool accumulate, int32_t *dev_status, void *stream,
                             const char *what) {
  if (m < 0 || n < 0 || lda < 0 || ldb < 0 || check_groups(num_experts) != FME_OK) return FME_ERR_INVALID_ARGUMENT;
  if (m % 256 != 0 || m == 0 || n % 256 != 0 || n == 0 || lda % 128 != 0 || ldb % 128 != 0)
    return FME_ERR_UNSUPPORTED_SHAPE;
  if (lda > (int64_t(1) << 31) - 1 || ldb > (int64_t(1) << 31) - 1 || m > 65536 || n > 65536)
    return FME_ERR_UNSUPPORTED_SHAPE;
  if (!padded_offsets || !y) return FME_ERR_INVALID_ARGUMENT;
  if (!aligned16(y) || !aligned16(padded_offsets)) return FME_ERR_MISALIGNED;
  const bool has_positions = lda > 0 && ldb > 0;
  if (has_positions) {
    if (!a_codes || !a_sf || !b_codes || !b_sf) return FME_ERR_INVALID_ARGUMENT;
    if (!aligned16(a_codes) || !aligned16(a_sf) || !aligned16(b_codes) || !aligned16(b_sf))
      return FME_ERR_MISALIGNED;
  }
  int sms = 0;
  fme_status st = current_device(&sms);
  if (st != FME_OK) return st;
  fme::LaunchGemm a{};
  a.kind = fme::GemmKind::kWgradMxfp8;
  // With no positions at all every expert is empty: the maps are never used, so
  // point them at a small dummy extent of y (always at least 256 x 256 x 2 bytes).
  const void *abase = has_positions ? static_cast<const void *>(a_codes) : y;
  const void *bbase = has_positions ? static_cast<const void *>(b_codes) : y;
  const void *sabase = has_positions ? static_cast<const void *>(a_sf) : y;
  const void *sbbase = has_positions ? static_cast<const void *>(b_sf) : y;
  const int64_t lda_e = has_positions ? lda : 128, ldb_e = has_positions ? ldb : 128;
  if ((st = encode_u8_2d(&a.map_a, abase, lda_e, has_positions ? m : 128, lda_e, 128)) != FME_OK) return st;
  if ((st = encode_u8_2d(&a.map_b, bbase, ldb_e, has_positions ? n : 128, ldb_e, 128)) != FME_OK) return st;
  if ((st = encode_scales_2d(&a.map_sfa, sabase, has_positions ? m / 128 : 1, (lda_e / 128) * 512, 1, 1)) != FME_OK)
    return st;
  if ((st = encode_scales_2d(&a.map_sfb, sbbase, has_positions ? n / 128 : 2, (ldb_e / 128) * 512, 1, 2)) != FME_OK)
    return st;
  // dW [num_experts * m x n] bf16 for bulk stores (the fp32 accumulate writes with plain stores)
  if (!accumulate && (st = encode_bf16_out(&a.map_y, y, n, static_cast<uint64_t>(num_experts) * m)) != FME_OK)
    return st;
  a.offsets = padded_offsets;
  a.num_experts = num_experts;
  a.m = m;
  a.n = n;
  a.k = 0;
  a.lda = lda;
  a.ldb = ldb;
  a.y = y;
  a.accumulate = accumulate;
  a.status = dev_status;
  a.num_sms = sms;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t err = fme::launch_grouped_gemm(a);
  return err == cudaSuccess ? FME_OK : cuda_fail(err, what);
}

fme_status grouped_gemm_wgrad_mxfp8(const uint8_t *a_codes, const uint8_t *a_sf, int64_t lda,
                                    const uint8_t *b_codes, const uint8_t *b_sf, int64_t ldb,
                                    const int32_t *padded_offsets, int32_t num_experts, int64_t m, int64_t n,
                                    void *y, int32_t *dev_status, void *stream) {
  return wgrad_call(a_codes, a_sf, lda, b_codes, b_sf, ldb, padded_offsets, num_experts, m, n, y, false, dev_status,
                    stream, "grouped_gemm_wgrad_mxfp8 launch");
}

fme_status grouped_gemm_wgrad_mxfp8_accumulate(const uint8_t *a_codes, const uint8_t *a_sf, int64_t lda,
                                               const uint8_t *b_codes, const uint8_t *b_sf, int64_t ldb,
                                               const int32_t *padded_offsets, int32_t num_experts, int64_t m,
                                               int64_t n, float *dw_acc, int32_t *dev_status, void *stream) {
  return wgrad_call(a_codes, a_sf, lda, b_codes, b_sf, ldb, padded_offsets, num_experts, m, n, dw_acc, true,
                    dev_status, stream, "grouped_gemm_wgrad_mxfp8_accumulate launch");
}

}  // extern "C"

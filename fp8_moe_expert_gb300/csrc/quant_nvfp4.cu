// quant_nvfp4.cu -- NVFP4 per-token quantizer (the forward's NVFP4 variant).
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1: bf16
// values become FP4 E2M1 codes with an FP8 E4M3 scale per 16-value block along K
// and an FP32 scale per token; the quantizer must use IEEE-compliant division.
// Per row: S = amax/2688, sb = E4M3(amax_b / fl32(6 S)), e = fl32(dec(sb) S),
// q = E2M1(x / e), all divisions correctly rounded (__fdiv_rn), all conversions
// round-to-nearest-even with saturation.
//
// One warp owns one row.  Lane l holds elements [256 c + 8 l, 256 c + 8 l + 8) of
// every 256-wide chunk c in registers (one 16-byte load per chunk), so the row
// is read from HBM once: the row amax is a warp max-reduction, a 16-block spans
// a lane pair (one shuffle), codes leave as one 4-byte store per lane per chunk
// (128 contiguous bytes per warp) and the four scales of four consecutive blocks
// leave as one 4-byte store into the tiled scale layout.
#include "fme_device.cuh"
#include "fme_launch.h"

namespace fme {

__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(code);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
}

// Two E2M1 codes: `lo` in bits 0..3, `hi` in bits 4..7.
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

template <int NCH>
__global__ void __launch_bounds__(128) nvfp4_pertoken_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                             int k, const int32_t *__restrict__ offsets,
                                                             int num_groups, uint8_t *__restrict__ codes,
                                                             uint8_t *__restrict__ sf,
                                                             float *__restrict__ row_scale, int32_t *status) {
  __shared__ GroupTable groups;
  __shared__ int ok_flag;
  if (!load_groups(groups, offsets, num_groups, rows, &ok_flag)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, kDevBadOffsets);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t c4 = ((k / 16) + 3) & ~3;

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); row < rows;
       row += static_cast<int64_t>(gridDim.x) * warps) {
    const uint16_t *xr = x + row * k;
    uint4 v[NCH];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int col = c * 256 + lane * 8;
      if (col < k)
        v[c] = __ldcs(reinterpret_cast<const uint4 *>(xr + col));
      else
        v[c] = make_uint4(0, 0, 0, 0);
    }
    // row amax (|x| as bits: bf16 magnitudes order like integers)
    uint32_t amax_bits = 0;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax_bits = max(amax_bits, w[i] & 0x7FFFu);
        amax_bits = max(amax_bits, (w[i] >> 16) & 0x7FFFu);
      }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, s));
    const float amax = bf16_bits_to_float(amax_bits);
    const float s_t = (amax_bits == 0) ? 0.0f : __fdiv_rn(amax, 2688.0f);
    const float d = __fmul_rn(6.0f, s_t);

    // padded row of the scale layout
    const int g = find_group(groups.off, num_groups, row);
    const int64_t prow = 128 * static_cast<int64_t>(groups.tiles[g]) + (row - groups.off[g]);
    uint8_t *codes_row = codes + row * (k / 2);

#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int col = c * 256 + lane * 8;
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
      uint32_t bmax = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bmax = max(bmax, w[i] & 0x7FFFu);
        bmax = max(bmax, (w[i] >> 16) & 0x7FFFu);
      }
      bmax = max(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 1));
      uint32_t sb = 0;
      if (bmax != 0) sb = e4m3_code(__fdiv_rn(bf16_bits_to_float(bmax), d));
      uint32_t packed = 0;
      if (sb != 0) {
        const float e = __fmul_rn(e4m3_value(sb), s_t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __fdiv_rn(bf16_bits_to_float(w[i] & 0xFFFFu), e);
          const float hi = __fdiv_rn(bf16_bits_to_float(w[i] >> 16), e);
          packed |= e2m1_pair(lo, hi) << (8 * i);
        }
      }
      if (col < k) *reinterpret_cast<uint32_t *>(codes_row + col / 2) = packed;
      // scales: block (c*16 + lane/2) is held by the even lane of each pair; lanes
      // 0, 8, 16, 24 gather four consecutive blocks and store them as one word.
      const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
      const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sb, 4);
      const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sb, 6);
      if ((lane & 7) == 0 && col < k) {
        const int64_t cb = c * 16 + lane / 2;
        const uint32_t word = sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
        *reinterpret_cast<uint32_t *>(sf + sf_offset(prow, cb, c4)) = word;
      }
    }
    if (lane == 0) row_scale[row] = s_t;
  }
}

template <int NCH>
static cudaError_t launch_nvfp4(const LaunchNvfp4 &a) {
  const int threads = 128;
  const int64_t blocks_needed = (a.rows + 3) / 4;
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 16;
  const int blocks = static_cast<int>(blocks_needed < cap ? (blocks_needed > 0 ? blocks_needed : 1) : cap);
  nvfp4_pertoken_kernel<NCH><<<blocks, threads, 0, a.stream>>>(
      static_cast<const uint16_t *>(a.x), a.rows, static_cast<int>(a.k), a.offsets, a.num_groups, a.codes, a.sf,
      a.row_scale, a.status);
  return cudaGetLastError();
}

cudaError_t launch_quantize_nvfp4(const LaunchNvfp4 &a) {
  const int nch = static_cast<int>((a.k + 255) / 256);
  if (nch <= 1) return launch_nvfp4<1>(a);
  if (nch <= 2) return launch_nvfp4<2>(a);
  if (nch <= 4) return launch_nvfp4<4>(a);
  if (nch <= 8) return launch_nvfp4<8>(a);
  if (nch <= 12) return launch_nvfp4<12>(a);
  if (nch <= 16) return launch_nvfp4<16>(a);
  if (nch <= 20) return launch_nvfp4<20>(a);
  if (nch <= 24) return launch_nvfp4<24>(a);
  if (nch <= 28) return launch_nvfp4<28>(a);
  return launch_nvfp4<32>(a);
}

}  // namespace fme

// quant_nvfp4.cu -- NVFP4 per-token quantizer (the forward's NVFP4 variant).
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1: bf16
// values become FP4 E2M1 codes with an FP8 E4M3 scale per 16-value block along K
// and an FP32 scale per token; the quantizer must use IEEE-compliant division.
// Per row: S = amax/2688, sb = E4M3(amax_b / fl32(6 S)), e = fl32(dec(sb) S),
// q = E2M1(x / e), all divisions correctly rounded (__fdiv_rn), all conversions
// round-to-nearest-even with saturation.
//
// One to four warps own one row (rows longer than 2048 values are split).  Lane
// l of a warp holds elements [256 c + 8 l, 256 c + 8 l + 8) of each 256-wide chunk
// c it owns in registers (one 16-byte load per chunk), so the row is read from
// HBM once: the row amax is a warp max-reduction (plus a shared-memory exchange
// between the row's warps), a 16-block spans a lane pair (one shuffle), codes
// leave as one 4-byte store per lane per chunk (128 contiguous bytes per warp)
// and the four scales of four consecutive blocks leave as one 4-byte store into
// the tiled scale layout.  The element codes come from the correctly rounded
// quotient fl32(x/e), found without a division unless the quotient sits next to
// an E2M1 rounding boundary (see e2m1_codes_of_quotients).
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

// Per-halfword unsigned max of two words of packed bf16 magnitudes.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest |x| of the 8 bf16 in a uint4, as bf16 magnitude bits.
__device__ __forceinline__ uint32_t amax8_bits(const uint4 &v) {
  const uint32_t m = max_u16x2(max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               max_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

// Two E2M1 codes: `lo` in bits 0..3, `hi` in bits 4..7.
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// E2M1 codes of the correctly rounded quotients fl32(x_i/e) of 8 bf16 values
// (4 words, element 2i in the low half of word i), packed two per byte with the
// even element in the low nibble, without dividing unless a quotient sits next
// to a rounding boundary of the E2M1 grid.
//
// With r an approximate reciprocal of a normal fp32 e (rcp.approx: within 2^-22
// relative), q = fl32(x r) differs from the exact x/e by less than 2^-21.7
// relative, and Q = fl32(x/e) by less than 2^-24, so Q lies strictly between
// fl32(q (1 - 2^-19)) and fl32(q (1 + 2^-19)).  Rounding to the E2M1 grid is
// monotone in |v| (same sign throughout), so when both ends round to the same
// code, Q does too.  If that fails for any of the 8 values (a quotient within
// about 2^-19 of a grid midpoint, e.g. an exact tie), all 8 codes come from the
// IEEE quotients themselves.  Quotients far below 0.25 round to (signed) zero on
// every path.  The result is always the codes of fl32(x/e).  Pairs go through
// the packed f32x2 multiplier.
__device__ __forceinline__ uint32_t e2m1_codes_of_quotients(const uint32_t (&w)[4], float e, float r,
                                                            bool normal_e) {
  constexpr float kBelow = 1.0f - 1.0f / 524288.0f;  // 1 - 2^-19, exact in fp32
  constexpr float kAbove = 1.0f + 1.0f / 524288.0f;  // 1 + 2^-19
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    const float2 q = __fmul2_rn(x, make_float2(r, r));
    const float2 a = __fmul2_rn(q, make_float2(kBelow, kBelow));
    const float2 b = __fmul2_rn(q, make_float2(kAbove, kAbove));
    lo[i] = e2m1_pair(a.x, a.y);
    hi[i] = e2m1_pair(b.x, b.y);
  }
  const uint32_t lo4 = __byte_perm(__byte_perm(lo[0], lo[1], 0x0040), __byte_perm(lo[2], lo[3], 0x0040), 0x5410);
  const uint32_t hi4 = __byte_perm(__byte_perm(hi[0], hi[1], 0x0040), __byte_perm(hi[2], hi[3], 0x0040), 0x5410);
  if (normal_e && lo4 == hi4) return lo4;
  uint32_t exact = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x0 = __uint_as_float(w[i] << 16);
    const float x1 = __uint_as_float(w[i] & 0xFFFF0000u);
    exact |= e2m1_pair(__fdiv_rn(x0, e), __fdiv_rn(x1, e)) << (8 * i);
  }
  return exact;
}

__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// Row split: WPR warps share one row; warp w of the row takes chunks w, w + WPR,
// ... (NCH of them), so every warp keeps at most 8 chunks (64 registers of data)
// in flight and the SM runs more warps.  The row amax is combined through shared
// memory behind a named barrier of the row's warps (slot parity alternates per
// row, so one barrier per row suffices).
constexpr int kNvThreads = 256;

__device__ __forceinline__ void row_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int NCH, int WPR>
__global__ void __launch_bounds__(kNvThreads, 3) nvfp4_pertoken_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                    int k, const int32_t *__restrict__ offsets,
                                                                    int num_groups, uint8_t *__restrict__ codes,
                                                                    uint8_t *__restrict__ sf,
                                                                    float *__restrict__ row_scale, int32_t *status) {
  constexpr int kRowsPerCta = (kNvThreads / 32) / WPR;
  __shared__ GroupTable groups;
  __shared__ int ok_flag;
  __shared__ uint32_t partial[2][kRowsPerCta][WPR];
  if (!load_groups(groups, offsets, num_groups, rows, &ok_flag)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, kDevBadOffsets);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int slot = warp / WPR;  // row slot of this CTA
  const int wr = warp % WPR;    // part of the row
  const int64_t c4 = ((k / 16) + 3) & ~3;
  int parity = 0;

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + slot; row < rows;
       row += static_cast<int64_t>(gridDim.x) * kRowsPerCta, parity ^= 1) {
    const uint16_t *xr = x + row * k;
    uint4 v[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int col = (wr + WPR * j) * 256 + lane * 8;
      if (col < k)
        v[j] = __ldcs(reinterpret_cast<const uint4 *>(xr + col));
      else
        v[j] = make_uint4(0, 0, 0, 0);
    }
    // per-chunk lane amax (|x| as bits: bf16 magnitudes order like integers), then row amax
    uint32_t lane_max[NCH];
    uint32_t amax_bits = 0;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      lane_max[j] = amax8_bits(v[j]);
      amax_bits = max(amax_bits, lane_max[j]);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, s));
    if (WPR > 1) {
      if (lane == 0) partial[parity][slot][wr] = amax_bits;
      row_barrier(1 + slot, WPR * 32);
#pragma unroll
      for (int i = 0; i < WPR; ++i) amax_bits = max(amax_bits, partial[parity][slot][i]);
    }
    const float amax = bf16_bits_to_float(amax_bits);
    const float s_t = (amax_bits == 0) ? 0.0f : __fdiv_rn(amax, 2688.0f);
    const float d = __fmul_rn(6.0f, s_t);

    // padded row of the scale layout; lanes 0, 8, 16, 24 store the scales of
    // blocks 16 c + lane/2 .. +3, i.e. tile 4 c + lane/8 of this row
    const int g = find_group(groups.off, num_groups, row);
    const int64_t prow = 128 * static_cast<int64_t>(groups.tiles[g]) + (row - groups.off[g]);
    uint8_t *codes_row = codes + row * (k / 2);
    uint8_t *sf_lane = sf + sf_offset(prow, 4 * (lane >> 3), c4);

#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = wr + WPR * j;
      const int col = c * 256 + lane * 8;
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      const uint32_t bmax = max(lane_max[j], __shfl_xor_sync(0xFFFFFFFFu, lane_max[j], 1));
      uint32_t sb = 0;
      if (bmax != 0) sb = e4m3_code(__fdiv_rn(bf16_bits_to_float(bmax), d));
      uint32_t packed = 0;
      if (sb != 0) {
        const float e = __fmul_rn(e4m3_value(sb), s_t);
        const bool normal_e = e >= 1.17549435e-38f;  // reciprocal finite and accurate
        packed = e2m1_codes_of_quotients(w, e, rcp_approx(e), normal_e);
      }
      if (col < k) *reinterpret_cast<uint32_t *>(codes_row + col / 2) = packed;
      // scales: block (16 c + lane/2) is held by the even lane of each pair; lanes
      // 0, 8, 16, 24 gather four consecutive blocks and store them as one word.
      const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
      const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sb, 4);
      const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sb, 6);
      if ((lane & 7) == 0 && col < k) {
        const uint32_t word = sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
        *reinterpret_cast<uint32_t *>(sf_lane + c * 2048) = word;
      }
    }
    if (lane == 0 && wr == 0) row_scale[row] = s_t;
  }
}

template <int NCH, int WPR>
static cudaError_t launch_nvfp4(const LaunchNvfp4 &a) {
  constexpr int rows_per_cta = (kNvThreads / 32) / WPR;
  const int64_t blocks_needed = (a.rows + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 8;
  const int blocks = static_cast<int>(blocks_needed < cap ? (blocks_needed > 0 ? blocks_needed : 1) : cap);
  nvfp4_pertoken_kernel<NCH, WPR><<<blocks, kNvThreads, 0, a.stream>>>(
      static_cast<const uint16_t *>(a.x), a.rows, static_cast<int>(a.k), a.offsets, a.num_groups, a.codes, a.sf,
      a.row_scale, a.status);
  return cudaGetLastError();
}

// Chunks of 256 values per row: up to 8 per warp, rows of more than 8 chunks
// are split over 2 or 4 warps (k <= 8192 = 32 chunks).
cudaError_t launch_quantize_nvfp4(const LaunchNvfp4 &a) {
  const int chunks = static_cast<int>((a.k + 255) / 256);
  if (chunks <= 1) return launch_nvfp4<1, 1>(a);
  if (chunks <= 2) return launch_nvfp4<2, 1>(a);
  if (chunks <= 4) return launch_nvfp4<4, 1>(a);
  if (chunks <= 8) return launch_nvfp4<8, 1>(a);
  if (chunks <= 16) return launch_nvfp4<8, 2>(a);
  return launch_nvfp4<8, 4>(a);
}

}  // namespace fme

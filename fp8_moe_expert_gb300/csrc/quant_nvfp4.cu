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
// l of a warp holds the 16-value block l of each 512-wide chunk it owns in
// registers (two 16-byte loads per chunk), so the row is read from HBM once:
// the row amax is a warp max-reduction (plus a shared-memory exchange between
// the row's warps), each block's amax, scale, reciprocal and codes stay in one
// lane, codes leave as one 8-byte store per lane per chunk (256 contiguous bytes
// per warp) and the four scales of four consecutive blocks leave as one 4-byte
// store into the tiled scale layout.  The element codes come from the correctly
// rounded quotient fl32(x/e), found without a division unless the quotient sits
// next to an E2M1 rounding boundary (see e2m1_block_codes).
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

// max(|a|, |b|) per bf16 half (sign bits hold the xor of the input signs).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest |x| of 16 bf16 values (two uint4), as bf16 magnitude bits.
__device__ __forceinline__ uint32_t amax16_bits(const uint4 &a, const uint4 &b) {
  const uint32_t m = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(a.x, a.y), absmax_bf16x2(a.z, a.w)),
                                   absmax_bf16x2(absmax_bf16x2(b.x, b.y), absmax_bf16x2(b.z, b.w)));
  return max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
}

// Two E2M1 codes: `lo` in bits 0..3, `hi` in bits 4..7.
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// E2M1 codes of the correctly rounded quotients fl32(x_i/e) of the 16 bf16 values
// of one block (8 words, element 2i in the low half of word i), packed two per
// byte with the even element in the low nibble, without dividing unless a
// quotient sits next to a rounding boundary of the E2M1 grid.
//
// With r an approximate reciprocal of a normal fp32 e (rcp.approx: within 2^-22
// relative), q = fl32(x r) differs from the exact x/e by less than 2^-21.7
// relative, and Q = fl32(x/e) by less than 2^-24, so Q lies strictly between
// fl32(q (1 - 2^-19)) and fl32(q (1 + 2^-19)).  Rounding to the E2M1 grid is
// monotone in |v| (same sign throughout), so when both ends round to the same
// code, Q does too.  If that fails for any of the 16 values (a quotient within
// about 2^-19 of a grid midpoint, e.g. an exact tie), all 16 codes come from the
// IEEE quotients themselves.  Quotients far below 0.25 round to (signed) zero on
// every path.  The result is always the codes of fl32(x/e).  Pairs go through
// the packed f32x2 multiplier.
__device__ __forceinline__ uint2 e2m1_block_codes(const uint32_t (&w)[8], float e, float r, bool normal_e) {
  constexpr float kBelow = 1.0f - 1.0f / 524288.0f;  // 1 - 2^-19, exact in fp32
  constexpr float kAbove = 1.0f + 1.0f / 524288.0f;  // 1 + 2^-19
  uint32_t lo[8];
  uint32_t diff = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 x = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    const float2 q = __fmul2_rn(x, make_float2(r, r));
    const float2 a = __fmul2_rn(q, make_float2(kBelow, kBelow));
    const float2 b = __fmul2_rn(q, make_float2(kAbove, kAbove));
    lo[i] = e2m1_pair(a.x, a.y);
    diff |= lo[i] ^ e2m1_pair(b.x, b.y);
  }
  uint2 out;
  out.x = __byte_perm(__byte_perm(lo[0], lo[1], 0x0040), __byte_perm(lo[2], lo[3], 0x0040), 0x5410);
  out.y = __byte_perm(__byte_perm(lo[4], lo[5], 0x0040), __byte_perm(lo[6], lo[7], 0x0040), 0x5410);
  if (normal_e && diff == 0) return out;
  uint32_t ex[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    ex[i] = e2m1_pair(__fdiv_rn(__uint_as_float(w[i] << 16), e), __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), e));
  out.x = __byte_perm(__byte_perm(ex[0], ex[1], 0x0040), __byte_perm(ex[2], ex[3], 0x0040), 0x5410);
  out.y = __byte_perm(__byte_perm(ex[4], ex[5], 0x0040), __byte_perm(ex[6], ex[7], 0x0040), 0x5410);
  return out;
}

// Row split: WPR warps share one row; warp w of the row takes chunks w, w + WPR,
// ... (NCH of them, 512 values each; lane l owns the 16-value block l of a
// chunk), so every warp keeps at most 4 chunks (64 registers of data) in flight.
// The row amax is combined through shared memory behind a named barrier of the
// row's warps (slot parity alternates per row, so one barrier per row suffices).
constexpr int kNvThreads = 256;

__device__ __forceinline__ void row_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int NCH, int WPR>
__global__ void __launch_bounds__(kNvThreads, 3) nvfp4_pertoken_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                       int k, const int32_t *__restrict__ offsets,
                                                                       int num_groups, uint8_t *__restrict__ codes,
                                                                       uint8_t *__restrict__ sf,
                                                                       float *__restrict__ row_scale,
                                                                       int32_t *status) {
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
    uint4 v[NCH][2];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int col = (wr + WPR * j) * 512 + lane * 16;
      if (col < k) {
        v[j][0] = __ldcs(reinterpret_cast<const uint4 *>(xr + col));
        v[j][1] = __ldcs(reinterpret_cast<const uint4 *>(xr + col + 8));
      } else {
        v[j][0] = make_uint4(0, 0, 0, 0);
        v[j][1] = make_uint4(0, 0, 0, 0);
      }
    }
    // block amax per chunk (|x| as bits: bf16 magnitudes order like integers), then row amax
    uint32_t bmax[NCH];
    uint32_t amax_bits = 0;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      bmax[j] = amax16_bits(v[j][0], v[j][1]);
      amax_bits = max(amax_bits, bmax[j]);
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

    // padded row of the scale layout; lanes 0, 4, .., 28 store the scales of
    // blocks 32 c + lane .. +3, i.e. tile 8 c + lane/4 of this row
    const int g = find_group(groups.off, num_groups, row);
    const int64_t prow = 128 * static_cast<int64_t>(groups.tiles[g]) + (row - groups.off[g]);
    uint8_t *codes_row = codes + row * (k / 2);
    uint8_t *sf_lane = sf + sf_offset(prow, 4 * (lane >> 2), c4);

#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = wr + WPR * j;
      const int col = c * 512 + lane * 16;
      const uint32_t w[8] = {v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w,
                             v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w};
      uint32_t sb = 0;
      if (bmax[j] != 0) sb = e4m3_code(__fdiv_rn(bf16_bits_to_float(bmax[j]), d));
      uint2 packed = make_uint2(0, 0);
      if (sb != 0) {
        const float e = __fmul_rn(e4m3_value(sb), s_t);
        const bool normal_e = e >= 1.17549435e-38f;  // reciprocal finite and accurate
        packed = e2m1_block_codes(w, e, rcp_approx(e), normal_e);
      }
      if (col < k) *reinterpret_cast<uint2 *>(codes_row + col / 2) = packed;
      // scales: lanes 4g .. 4g+3 hold blocks 32 c + 4g .. +3; lane 4g stores them as one word
      const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sb, 1);
      const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
      const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sb, 3);
      if ((lane & 3) == 0 && col < k) {
        const uint32_t word = sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
        *reinterpret_cast<uint32_t *>(sf_lane + c * 4096) = word;
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

// Chunks of 512 values per row: up to 4 per warp, rows of more than 4 chunks are
// split over 2 or 4 warps (k <= 8192 = 16 chunks).
cudaError_t launch_quantize_nvfp4(const LaunchNvfp4 &a) {
  const int chunks = static_cast<int>((a.k + 511) / 512);
  if (chunks <= 1) return launch_nvfp4<1, 1>(a);
  if (chunks <= 2) return launch_nvfp4<2, 1>(a);
  if (chunks <= 4) return launch_nvfp4<4, 1>(a);
  if (chunks <= 8) return launch_nvfp4<4, 2>(a);
  return launch_nvfp4<4, 4>(a);
}

}  // namespace fme

// quant_nvfp4.cu -- NVFP4 per-token quantizer (the forward's NVFP4 variant).
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1: bf16
// values become FP4 E2M1 codes with an FP8 E4M3 scale per 16-value block along K
// and an FP32 scale per token; the quantizer must use IEEE-compliant division.
// Per row: S = amax/2688, sb = E4M3(amax_b / fl32(6 S)), e = fl32(dec(sb) S),
// q = E2M1(x / e), all divisions correctly rounded (__fdiv_rn), all conversions
// round-to-nearest-even with saturation.
//
// One CTA quantizes one row at a time; each thread owns R (1 or 2) of the row's
// 16-value blocks, t and t + T.  Rows stream through a ring of shared-memory
// stages filled by bulk asynchronous copies (one cp.async.bulk per row,
// completing on the stage's mbarrier) issued several rows ahead by thread 0, so
// the HBM reads stay in flight while the CTA computes.  Per row: every thread
// reads its blocks once from shared memory, the row amax is a warp max-reduction
// plus one CTA barrier, then each thread derives its block scales and codes in
// registers.  Codes leave as 8-byte stores (256 contiguous bytes per warp) and
// the scales of four consecutive blocks as one 4-byte store into the tiled scale
// layout.  Block scales and element codes come from the correctly rounded
// quotients: block scales from a bracket that divides only when a quotient sits
// next to an E4M3 rounding boundary (e4m3_quotient_code), element codes from one
// exact correction step that never divides (e2m1_block_codes).
#include <type_traits>

#include "fme_device.cuh"
#include "fme_launch.h"

namespace fme {

__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// Value of a non-negative, finite E4M3 code.  The code shifted into the top of an
// fp32 (exponent field = E4M3 exponent field, mantissa = its 3 bits) is the value
// times 2^-120, also for the E4M3 subnormals (fp32 subnormals then); the
// multiply by 2^120 is exact.
__device__ __forceinline__ float e4m3_value(uint32_t code) { return __uint_as_float(code << 20) * 0x1p120f; }

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

// Two E2M1 codes (one byte) of the IEEE quotients fl32(lo/e), fl32(hi/e).
__device__ __forceinline__ uint32_t e2m1_pair_exact(uint32_t w, float e) {
  return e2m1_pair(__fdiv_rn(__uint_as_float(w << 16), e), __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), e));
}

// The E2M1 codes of four pairs (v[2i], v[2i+1]) packed as bytes 0..3 of a word,
// the pair's first value in the byte's low nibble: four conversions into byte
// registers and one vector move.
__device__ __forceinline__ uint32_t e2m1_x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Bytes 0..3 of a, b, c, d (each holding two codes in its low byte) as one word.
__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Smallest decode scale e whose blocks are coded without a division.  Below it the
// residual of the correction step (e2m1_step_codes) could lose bits in the
// subnormal range; such blocks (block scales far below any real data's) divide.
constexpr float kE2M1StepMinScale = 0x1p-76f;

// E2M1 codes of the correctly rounded quotients fl32(x_i/e) of the 16 bf16 values
// of one block (8 words, element 2i in the low half of word i), packed two per
// byte with the even element in the low nibble, without a division.
//
// One correction step on fused multiply-adds after the reciprocal product
// (Markstein's division refinement): with r = rcp.approx(e) (PTX ISA: at most one
// ulp from 1/e), q = fl32(x r), rho = fl32(x - q e), Q = fl32(q + rho r).  Q is
// the IEEE quotient fl32(x/e) for every bf16 x with x/e in [2^-4, 8] and every
// e >= 2^-76 made from a bf16 row amax and an E4M3 block scale, whatever r is
// within four ulps of 1/e: checked exhaustively on the CPU, every case bit for bit.
// Quotients below 2^-4 give a signed-zero code on both sides (|Q| stays far
// below the first E2M1 midpoint 0.25 and keeps x's sign).  Here the step runs
// negated, n = fl32(x (-r)) = -q, rho = fl32(n e + x), t = fl32(rho (-r) + n) =
// -Q, and the codes of t get their sign bits flipped: for x = -0 the plain form
// ends in (+0) + (-0) = +0 where the IEEE quotient is -0, the negated one in
// (-0) + (+0) = +0 = -(-0).  Pairs go through the packed f32x2 pipe.  Valid for
// e >= kE2M1StepMinScale (e2m1_block_codes below adds the test).
__device__ __forceinline__ uint2 e2m1_step_codes(const uint32_t (&w)[8], float e) {
  const float nr = -rcp_approx(e);
  const float2 nr2 = make_float2(nr, nr);
  const float2 e2 = make_float2(e, e);
  float t[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 x = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    const float2 n = __fmul2_rn(x, nr2);
#ifdef FME_TEST_APPROX_DIVIDE
    // Test build only (tests/test_gpu_division_control.py): the approximate
    // quotient x * rcp.approx(e) of a fast divide, without the correction step.
    const float2 q = n;
    (void)e2;
#else
    const float2 rho = __ffma2_rn(n, e2, x);
    const float2 q = __ffma2_rn(rho, nr2, n);
#endif
    t[2 * i] = q.x;
    t[2 * i + 1] = q.y;
  }
  const float(&t0)[8] = *reinterpret_cast<const float(*)[8]>(&t[0]);
  const float(&t1)[8] = *reinterpret_cast<const float(*)[8]>(&t[8]);
  return make_uint2(e2m1_x8(t0) ^ 0x88888888u, e2m1_x8(t1) ^ 0x88888888u);
}

// The same codes for any e > 0: the correction step where it is exact, IEEE
// divisions below kE2M1StepMinScale.
__device__ __forceinline__ uint2 e2m1_block_codes(const uint32_t (&w)[8], float e) {
  if (!(e >= kE2M1StepMinScale)) {
    return make_uint2(pack4(e2m1_pair_exact(w[0], e), e2m1_pair_exact(w[1], e), e2m1_pair_exact(w[2], e),
                            e2m1_pair_exact(w[3], e)),
                      pack4(e2m1_pair_exact(w[4], e), e2m1_pair_exact(w[5], e), e2m1_pair_exact(w[6], e),
                            e2m1_pair_exact(w[7], e)));
  }
  return e2m1_step_codes(w, e);
}

// E4M3 code of the correctly rounded quotient fl32(v / d), v >= 0, with rd_lo /
// rd_hi an approximate reciprocal of d (rcp.approx; d normal) times 1 -+ 2^-19,
// rounded.  rd is within 2^-22 of 1/d relative, so fl32(v rd_lo) and fl32(v rd_hi)
// differ from v/d (1 -+ 2^-19) by less than 2^-22 + 2^-23 relative, while
// fl32(v/d) is within 2^-24 of v/d: the two products enclose fl32(v/d).  Rounding
// to E4M3 is monotone, so if both round to the same code (one cvt converts both),
// that is the code of fl32(v/d).  Otherwise (a quotient within about 2^-19 of an
// E4M3 midpoint: rare, E4M3 midpoints are far apart), or when d is not normal,
// the quotient is computed with an IEEE division.
__device__ __forceinline__ uint32_t e4m3_quotient_code(float v, float d, float rd_lo, float rd_hi, bool normal_d) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(__fmul_rn(v, rd_hi)), "f"(__fmul_rn(v, rd_lo)));
  const uint32_t lo = pair & 0xFFu;
  if (normal_d && lo == (static_cast<uint32_t>(pair) >> 8)) return lo;
  return e4m3_code(__fdiv_rn(v, d));
}

// S = fl32(amax / 2688) for a bf16 amax, without a division: q = fl32(amax r) with
// r = fl32(1/2688), then one correction step q + (amax - q 2688) r on fused
// multiply-adds (the residual is exact).  Equal to the IEEE quotient for every
// positive finite bf16 value (all 32639 checked, exactly, against correctly
// rounded division; the GPU tests repeat the check on the device).
__device__ __forceinline__ float per_token_scale(float amax) {
  constexpr float kInv = 1.0f / 2688.0f;
  const float q = __fmul_rn(amax, kInv);
  return __fmaf_rn(__fmaf_rn(-q, 2688.0f, amax), kInv, q);
}

constexpr int kNvMaxThreads = 256;         // threads per CTA: blocks per row / R, rounded up to warps
constexpr int kNvSmemBudget = 220 * 1024;  // shared memory aimed for per SM

// Shared-memory layout of the dynamic part: [stages x row][stages mbarriers]
// [G+1 group offsets][G+1 tile counts].
__host__ __device__ __forceinline__ size_t nv_smem_bytes(int stages, int64_t row_bytes, int num_groups) {
  return static_cast<size_t>(stages) * (row_bytes + 8) + 8 * static_cast<size_t>(num_groups + 1);
}

// SwiGLU of two bf16 words: gate (g.lo, g.hi) and up (u.lo, u.hi) -> the bf16 word
// (h.lo, h.hi), h = silu(g) * u rounded to bf16 (nearest even).
__device__ __forceinline__ uint32_t swiglu_word(uint32_t g, uint32_t u) {
  const float h0 = silu_times(__uint_as_float(g << 16), __uint_as_float(u << 16));
  const float h1 = silu_times(__uint_as_float(g & 0xFFFF0000u), __uint_as_float(u & 0xFFFF0000u));
  const __nv_bfloat162 h = __floats2bfloat162_rn(h0, h1);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint4 swiglu_uint4(const uint4 &g, const uint4 &u) {
  return make_uint4(swiglu_word(g.x, u.x), swiglu_word(g.y, u.y), swiglu_word(g.z, u.z), swiglu_word(g.w, u.w));
}

// kSwiGLU: the row is produced from a gate/up row [g (k values) | u (k values)]
// staged whole in shared memory: h = silu(g) * u rounded to bf16, optionally
// written to h_out, then quantized exactly as a bf16 input row would be.
template <int R, bool kSwiGLU, bool kGather>
__global__ void __launch_bounds__(kNvMaxThreads, 4)
    nvfp4_pertoken_kernel(const uint16_t *__restrict__ x, int64_t rows, int k, const int32_t *__restrict__ offsets,
                          int num_groups, uint8_t *__restrict__ codes, uint8_t *__restrict__ sf,
                          float *__restrict__ row_scale, uint16_t *__restrict__ h_out, int32_t *status,
                          int stages, const int32_t *__restrict__ gather, int gather_div, int64_t gather_limit,
                          const float *__restrict__ tensor_amax) {
  __shared__ int ok_flag;
  __shared__ int abort_flag;
  __shared__ uint32_t part[2][kNvMaxThreads / 32];  // per-warp amax of the row, double-buffered by row parity
  __shared__ int64_t sf_row_of[2];                   // byte offset of the row's scales (block 0) in sf
  extern __shared__ __align__(128) uint8_t nv_smem[];
  const uint32_t row_bytes = static_cast<uint32_t>(k) * (kSwiGLU ? 4u : 2u);  // staged input row
  const int64_t row_elems = kSwiGLU ? 2 * static_cast<int64_t>(k) : k;
  uint64_t *bars = reinterpret_cast<uint64_t *>(nv_smem + static_cast<size_t>(stages) * row_bytes);
  int32_t *g_off = reinterpret_cast<int32_t *>(bars + stages);
  int32_t *g_tiles = g_off + num_groups + 1;
  if (!load_groups(g_off, g_tiles, offsets, num_groups, rows, &ok_flag)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, kDevBadOffsets);
    return;
  }
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int T = blockDim.x;
  const int nblk = k / 16;
  const int64_t first = blockIdx.x;
  const int64_t stride = gridDim.x;
  const int64_t c4 = (nblk + 3) & ~3;
  // i-th row this CTA quantizes
  auto row_at = [&](int64_t i) -> int64_t { return first + i * stride; };

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  // the gathered token of a gather entry (checked)
  auto token_of = [&](int32_t entry) -> int64_t {
    const int64_t g = entry / gather_div;
    if (g < 0 || g >= gather_limit) {
      report(status, kDevBadIndex);
      return 0;
    }
    return g;
  };
  // input row of output row r: r itself, or the gathered token
  auto src_of = [&](int64_t r) -> int64_t { return kGather ? token_of(__ldg(gather + r)) : r; };
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      const int64_t r = row_at(s);
      if (r >= rows) break;
      mbar_arrive_expect_tx(&bars[s], row_bytes);
      bulk_load(nv_smem + static_cast<size_t>(s) * row_bytes, x + src_of(r) * row_elems, row_bytes, &bars[s]);
    }
  }

  // lanes whose quad index is odd read the second 16 bytes of their block first,
  // so a quarter-warp's 16-byte reads cover all 32 banks
  const int swap = (tid >> 2) & 1;
  int i = 0, s = 0;
  uint32_t parity = 0;
  int g_cur = 0;  // thread 0: group of the current row (activations)
  // thread 0, gathering: the gather entry of the next row to refill, loaded one
  // row ahead so that its latency overlaps a row's work instead of delaying the
  // refill's copy
  int32_t next_entry = 0;
  if (kGather && tid == 0 && row_at(stages) < rows) next_entry = __ldg(gather + row_at(stages));
  int64_t row = row_at(0);
  for (; row < rows; ++i, row += stride) {
    const bool ok = mbar_wait(&bars[s], parity, &abort_flag, status);
    const uint8_t *buf = nv_smem + static_cast<size_t>(s) * row_bytes;
    uint4 a[R], b[R];
    uint32_t bmax[R];
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int blk = tid + j * T;
      a[j] = make_uint4(0, 0, 0, 0);
      b[j] = make_uint4(0, 0, 0, 0);
      if (ok && blk < nblk) {
        a[j] = *reinterpret_cast<const uint4 *>(buf + blk * 32 + 16 * swap);
        b[j] = *reinterpret_cast<const uint4 *>(buf + blk * 32 + 16 * (1 - swap));
        if (kSwiGLU) {
          const uint8_t *up = buf + 2 * static_cast<size_t>(k);
          a[j] = swiglu_uint4(a[j], *reinterpret_cast<const uint4 *>(up + blk * 32 + 16 * swap));
          b[j] = swiglu_uint4(b[j], *reinterpret_cast<const uint4 *>(up + blk * 32 + 16 * (1 - swap)));
          if (h_out != nullptr) {
            uint16_t *hb = h_out + row * k + blk * 16;
            *reinterpret_cast<uint4 *>(hb + 8 * swap) = a[j];
            *reinterpret_cast<uint4 *>(hb + 8 * (1 - swap)) = b[j];
          }
        }
      }
      bmax[j] = amax16_bits(a[j], b[j]);
      m = max(m, bmax[j]);
    }
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) part[i & 1][warp] = wmax;
    if (tid == 0) {
      // rows only increase here (first + i stride): move the group cursor forward
      while (g_cur + 1 < num_groups && g_off[g_cur + 1] <= row) ++g_cur;
      const int g = g_cur;
      const int64_t prow = 128 * static_cast<int64_t>(g_tiles[g]) + (row - g_off[g]);
      sf_row_of[i & 1] = sf_offset(prow, 0, c4);
    }
    if (__syncthreads_or(!ok)) break;  // every block of stage s is in registers: refill it
    if (tid == 0) {
      const int64_t next = row + stages * stride;
      if (next < rows) {
        const int64_t src = kGather ? token_of(next_entry) : next;
        fence_proxy_async_shared();
        mbar_arrive_expect_tx(&bars[s], row_bytes);
        bulk_load(nv_smem + static_cast<size_t>(s) * row_bytes, x + src * row_elems, row_bytes, &bars[s]);
        if (kGather && next + stride < rows) next_entry = __ldg(gather + next + stride);
      }
    }
    if (++s == stages) {
      s = 0;
      parity ^= 1u;
    }
    uint32_t amax_bits = __reduce_max_sync(0xFFFFFFFFu, lane < nwarps ? part[i & 1][lane] : 0u);
    if (tensor_amax != nullptr) amax_bits = __float_as_uint(*tensor_amax) >> 16;  // standard NVFP4: one scale
    uint8_t *sf_row = sf + sf_row_of[i & 1];
    uint8_t *codes_row = codes + row * (k / 2);
    const float amax = bf16_bits_to_float(amax_bits);
    const float s_t = (amax_bits == 0) ? 0.0f : per_token_scale(amax);
    const float d = __fmul_rn(6.0f, s_t);
    const bool normal_d = d >= 1.17549435e-38f;
    const float rd = rcp_approx(d);
    const float rd_lo = __fmul_rn(rd, 1.0f - 1.0f / 524288.0f);  // 1 - 2^-19, exact
    const float rd_hi = __fmul_rn(rd, 1.0f + 1.0f / 524288.0f);
    // Codes and scales of this thread's blocks.  step_all: every block of the row
    // takes the correction step, without a per-block test or branch (every e is at
    // least 2^-9 s_t, the smallest E4M3 value times s_t, so s_t >= 2^-67 puts every
    // e at or above 2^-76); 5-7% faster than the per-block test.
    auto code_blocks = [&](auto step_all) {
      // all R blocks' scales and codes first (independent chains the compiler can
      // interleave), then their stores and the warp-wide scale-word shuffles
      uint32_t sbs[R];
      uint2 packed[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        uint32_t sb = 0;
        if (bmax[j] != 0) sb = e4m3_quotient_code(bf16_bits_to_float(bmax[j]), d, rd_lo, rd_hi, normal_d);
        const uint32_t w[8] = {a[j].x, a[j].y, a[j].z, a[j].w, b[j].x, b[j].y, b[j].z, b[j].w};
        uint2 pk = make_uint2(0, 0);
        if constexpr (decltype(step_all)::value) {
          // sb = 0 (codes 0): the step runs on e = 1, harmlessly, and is discarded
          pk = e2m1_step_codes(w, sb != 0 ? __fmul_rn(e4m3_value(sb), s_t) : 1.0f);
          if (swap) pk = make_uint2(pk.y, pk.x);
          if (sb == 0) pk = make_uint2(0, 0);
        } else if (sb != 0) {
          pk = e2m1_block_codes(w, __fmul_rn(e4m3_value(sb), s_t));
          if (swap) pk = make_uint2(pk.y, pk.x);
        }
        sbs[j] = sb;
        packed[j] = pk;
      }
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int blk = tid + j * T;
        const uint32_t sb = sbs[j];
        if (blk < nblk) *reinterpret_cast<uint2 *>(codes_row + blk * 8) = packed[j];
        // scales: threads 4g .. 4g+3 hold blocks blk .. blk+3 (blk = 4g + jT); thread 4g
        // stores them as one word
        const uint32_t pair = __byte_perm(sb, __shfl_down_sync(0xFFFFFFFFu, sb, 1), 0x0040);
        const uint32_t word = __byte_perm(pair, __shfl_down_sync(0xFFFFFFFFu, pair, 2), 0x5410);  // lanes 4g
        if ((lane & 3) == 0 && blk < nblk) *reinterpret_cast<uint32_t *>(sf_row + (blk >> 2) * 512) = word;
      }
    };
    if (s_t >= 0x1p-67f) {
      code_blocks(std::true_type{});
    } else {
      code_blocks(std::false_type{});
    }
    if (tid == 0) row_scale[row] = s_t;
  }
  if (row < rows && tid == 0) {
    // gave up on a stage: wait (bounded) for the copies still in flight into this
    // CTA's shared memory before it exits
    const uint64_t t0 = globaltimer();
    for (int j = 0; j < stages && row_at(i + j) < rows; ++j) {
      while (!mbar_try_wait(&bars[s], parity) && globaltimer() - t0 < kDrainLimitNs) {
      }
      if (++s == stages) {
        s = 0;
        parity ^= 1u;
      }
    }
  }
}

// R = blocks per thread (1, 2 or 4, see launch_quantize_nvfp4); threads = blocks
// / R rounded up to warps.  CTAs per SM: as many as 1024 threads and the
// shared-memory budget allow with at least 3 stages each; stages: the rest of
// the budget, 3 to 16 rows.
template <int R, bool kSwiGLU, bool kGather>
static cudaError_t launch_nvfp4(const LaunchNvfp4 &a) {
  const int64_t nblk = a.k / 16;
  const int64_t row_bytes = a.k * (kSwiGLU ? 4 : 2);
  const int threads = static_cast<int>(((nblk + R - 1) / R + 31) / 32 * 32);
  const int64_t fixed = 1024 + 8 * (a.num_groups + 1);
  int per_sm = 1024 / threads;
  if (per_sm > 16) per_sm = 16;
  while (per_sm > 1 && per_sm * (static_cast<int64_t>(nv_smem_bytes(3, row_bytes, 0)) + fixed) > kNvSmemBudget)
    --per_sm;
  int64_t stages = (kNvSmemBudget / per_sm - fixed) / (row_bytes + 8);
  stages = stages < 3 ? 3 : (stages > 16 ? 16 : stages);
  const size_t smem = nv_smem_bytes(static_cast<int>(stages), row_bytes, a.num_groups);
  auto kernel = nvfp4_pertoken_kernel<R, kSwiGLU, kGather>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int64_t cap = static_cast<int64_t>(a.num_sms) * per_sm;
  const int blocks = static_cast<int>(a.rows < cap ? (a.rows > 0 ? a.rows : 1) : cap);
  kernel<<<blocks, threads, smem, a.stream>>>(static_cast<const uint16_t *>(a.x), a.rows, static_cast<int>(a.k),
                                              a.offsets, a.num_groups, a.codes, a.sf, a.row_scale,
                                              static_cast<uint16_t *>(a.h_out), a.status, static_cast<int>(stages),
                                              a.gather, a.gather_div, a.gather_limit, a.tensor_amax);
  return cudaGetLastError();
}

// max |x| over n bf16 values (n a multiple of 8) into *out (zeroed before): the
// bf16 maximum as an fp32 whose bits order like unsigned integers, so one
// atomicMax per CTA merges the CTAs' maxima.
__global__ void __launch_bounds__(256) tensor_amax_kernel(const uint16_t *__restrict__ x, int64_t n, float *out) {
  uint32_t m = 0;
  const int64_t words = n / 8;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < words;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(x) + w);
    m = max(m, amax16_bits(v, v));
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t v = threadIdx.x < (blockDim.x >> 5) ? wm[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int *>(out), v << 16);
  }
}

cudaError_t launch_quantize_nvfp4_pertensor(const LaunchNvfp4 &a, float *tensor_amax) {
  cudaError_t err = cudaMemsetAsync(tensor_amax, 0, sizeof(float), a.stream);
  if (err != cudaSuccess) return err;
  const int64_t words = a.rows * a.k / 8;
  const int64_t need = (words + 255) / 256;
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 8;
  const int blocks = static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
  tensor_amax_kernel<<<blocks, 256, 0, a.stream>>>(static_cast<const uint16_t *>(a.x), a.rows * a.k, tensor_amax);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  LaunchNvfp4 b = a;
  b.tensor_amax = tensor_amax;
  return launch_quantize_nvfp4(b);
}

// Two blocks per thread (measured on GB300: k = 2048 with 64 threads per CTA runs
// 8-14% faster than with 128, k = 7168 fastest with 224; three or four blocks per
// thread are slower).  The SwiGLU rows (twice the bytes per block) keep one block
// per thread up to 256 blocks, measured 4% faster there.
cudaError_t launch_quantize_nvfp4(const LaunchNvfp4 &a) {
  // the gathered variant is a kernel of its own, so the plain rows carry no gather code
  if (a.swiglu) return a.k / 16 > kNvMaxThreads ? launch_nvfp4<2, true, false>(a) : launch_nvfp4<1, true, false>(a);
  if (a.gather != nullptr) return launch_nvfp4<2, false, true>(a);
  // up to 2048 values per row, one warp per row (four blocks per thread): the row's
  // amax needs no barrier across warps (measured at k = 2048: 0.276 -> 0.249 ms for
  // 262144 rows, 0.236 -> 0.215 ms for 229376)
  return a.k <= 2048 ? launch_nvfp4<4, false, false>(a) : launch_nvfp4<2, false, false>(a);
}

}  // namespace fme

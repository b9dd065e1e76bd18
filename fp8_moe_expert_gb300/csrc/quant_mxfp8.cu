// quant_mxfp8.cu -- MXFP8 quantizers of the backward (row-wise and column-wise).
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1, paragraph
// on MXFP8 in the MoE backward: standard MXFP8, FP8 E4M3 values with an FP8
// E8M0 scale per block of 32.  Scale rule of the OCP MX v1.0 format the report
// cites: X = 2^(floor(log2 amax) - 8), code = clamp(floor(log2 amax) + 119, 0, 254).
// For a bf16 amax that is max(0, exponent field - 8), read straight from the
// bits; x / X is then one exact fp32 multiply by 2^(127 - code), so the fast
// division the pages allow for MXFP8 and a correctly rounded one give the same
// codes.  Elements convert with cvt.rn.satfinite (nearest even, saturating at 448).
//
// The SwiGLU backward of the gate/up projection (h = silu(g) * u, the activation
// between the two expert projections) is fused with the row-wise and column-wise
// quantization of its result d(gate_up) = [dg | du], the A operands of the gate/up
// data and weight gradients: dg = dh * u * sigma(g) * (1 + g * sigma(-g)),
// du = dh * g * sigma(g), each evaluated in fp32 and rounded to bf16 before it is
// quantized exactly as a bf16 input would be.
#include "fme_device.cuh"
#include "fme_launch.h"

namespace fme {

__device__ __forceinline__ uint32_t mx_code_from_bf16_amax(uint32_t amax_bits) {
  const int e = static_cast<int>((amax_bits >> 7) & 0xFF);
  return static_cast<uint32_t>(e > 8 ? e - 8 : 0);
}

// The round-up scale variant X = 2^ceil(log2(amax / 448)) (no element saturates):
// with 448 = 1.75 * 2^8 that is the exponent field minus 8, plus one when the
// significand is above 1.75 (fraction bits above 0x60); clamped at 0.
__device__ __forceinline__ uint32_t mx_code_ceil_from_bf16_amax(uint32_t amax_bits) {
  const int e = static_cast<int>((amax_bits >> 7) & 0xFF);
  const int c = e - 8 + ((amax_bits & 0x7Fu) > 0x60u ? 1 : 0);
  return static_cast<uint32_t>(c > 0 ? c : 0);
}

template <bool kCeil>
__device__ __forceinline__ uint32_t mx_code(uint32_t amax_bits) {
  return kCeil ? mx_code_ceil_from_bf16_amax(amax_bits) : mx_code_from_bf16_amax(amax_bits);
}

__device__ __forceinline__ float rcp_fast(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// (dg, du) of two elements: gate g, up u, upstream gradient dh, on the packed
// f32x2 pipe.  sigma(g) and sigma(-g) come from t = e^(-|g|) as (1 or t) / (1 + t),
// so neither is formed as 1 - sigma (no cancellation for large |g|) and
// e^(-|g|) never overflows.
__device__ __forceinline__ void swiglu_bwd_pair(float2 g, float2 u, float2 dh, float2 &dg, float2 &du) {
  const float2 s = make_float2(__expf(-0.5f * fabsf(g.x)), __expf(-0.5f * fabsf(g.y)));
  const float2 t = __fmul2_rn(s, s);
  const float2 r = make_float2(rcp_fast(1.0f + t.x), rcp_fast(1.0f + t.y));
  const float2 sig = __fmul2_rn(make_float2(g.x >= 0.0f ? 1.0f : t.x, g.y >= 0.0f ? 1.0f : t.y), r);
  const float2 sig_neg = __fmul2_rn(make_float2(g.x >= 0.0f ? t.x : 1.0f, g.y >= 0.0f ? t.y : 1.0f), r);
  du = __fmul2_rn(dh, __fmul2_rn(g, sig));
  dg = __fmul2_rn(__fmul2_rn(dh, u), __fmul2_rn(sig, __ffma2_rn(g, sig_neg, make_float2(1.0f, 1.0f))));
}

// Eight elements (one 16-byte word of g, u and dh each) -> the bf16 words of dg
// and du (nearest even).
__device__ __forceinline__ void swiglu_bwd_uint4(const uint4 &g, const uint4 &u, const uint4 &dh, uint4 &dg,
                                                 uint4 &du) {
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w}, hw[4] = {dh.x, dh.y, dh.z, dh.w};
  uint32_t ow_g[4], ow_u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 gf = make_float2(__uint_as_float(gw[i] << 16), __uint_as_float(gw[i] & 0xFFFF0000u));
    const float2 uf = make_float2(__uint_as_float(uw[i] << 16), __uint_as_float(uw[i] & 0xFFFF0000u));
    const float2 hf = make_float2(__uint_as_float(hw[i] << 16), __uint_as_float(hw[i] & 0xFFFF0000u));
    float2 dgf, duf;
    swiglu_bwd_pair(gf, uf, hf, dgf, duf);
    const __nv_bfloat162 bg = __floats2bfloat162_rn(dgf.x, dgf.y);
    const __nv_bfloat162 bu = __floats2bfloat162_rn(duf.x, duf.y);
    ow_g[i] = *reinterpret_cast<const uint32_t *>(&bg);
    ow_u[i] = *reinterpret_cast<const uint32_t *>(&bu);
  }
  dg = make_uint4(ow_g[0], ow_g[1], ow_g[2], ow_g[3]);
  du = make_uint4(ow_u[0], ow_u[1], ow_u[2], ow_u[3]);
}

// 2^(127 - code) as an fp32 (code in [0, 246] for bf16 inputs: always normal).
__device__ __forceinline__ float mx_inv_scale(uint32_t code) { return __uint_as_float((254u - code) << 23); }

// max(|a|, |b|) per bf16 half (sign bits hold the xor of the input signs).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Four E4M3 codes in value order, packed into a word by one vector move of two
// 16-bit conversion results.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
  uint32_t r;
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
      "mov.b32 %0, {h0, h1};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return r;
}

// Four values given as fp32 bit patterns (bf16 widened) times s (two packed
// multiplies, exact: s is a power of two) -> four E4M3 codes in that order.
__device__ __forceinline__ uint32_t e4m3x4_scaled(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, float s) {
  const float2 p = __fmul2_rn(make_float2(__uint_as_float(w0), __uint_as_float(w1)), make_float2(s, s));
  const float2 q = __fmul2_rn(make_float2(__uint_as_float(w2), __uint_as_float(w3)), make_float2(s, s));
  return e4m3x4(p.x, p.y, q.x, q.y);
}

// The two bf16 of each of words a, b (elements a.lo, a.hi, b.lo, b.hi) times s
// -> four E4M3 codes in element order.
__device__ __forceinline__ uint32_t e4m3x4_words(uint32_t a, uint32_t b, float s) {
  return e4m3x4_scaled(a << 16, a & 0xFFFF0000u, b << 16, b & 0xFFFF0000u, s);
}

// ---------------------------------------------------------------- row-wise --
// One warp per row; lane l handles 8 consecutive values of every 256-wide
// chunk, four lanes form a 32-block (two shuffles for its amax).  Codes leave as
// 8-byte stores (256 contiguous bytes per warp); lanes 0 and 16 each store four
// consecutive scales as one word of the tiled layout.  With `gather`, row r reads
// source row gather[r] / gather_div (grouped rows of routed tokens); an index
// outside [0, gather_limit) is reported and reads source row 0.
constexpr int kRowUnroll = 4;

template <bool kCeil>
__global__ void __launch_bounds__(256) mxfp8_rows_kernel(const uint16_t *__restrict__ x, int64_t rows, int cols,
                                                         const int32_t *__restrict__ offsets, int num_groups,
                                                         uint8_t *__restrict__ codes, uint8_t *__restrict__ sf,
                                                         int32_t *status, const int32_t *__restrict__ gather,
                                                         int gather_div, int64_t gather_limit) {
  __shared__ GroupTable groups;
  __shared__ int ok_flag;
  if (!load_groups(groups, offsets, num_groups, rows, &ok_flag)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, kDevBadOffsets);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t c4 = ((cols / 32) + 3) & ~3;

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); row < rows;
       row += static_cast<int64_t>(gridDim.x) * warps) {
    const int g = find_group(groups.off, num_groups, row);
    const int64_t prow = 128 * static_cast<int64_t>(groups.tiles[g]) + (row - groups.off[g]);
    int64_t src = row;
    if (gather) {
      src = __ldg(gather + row) / gather_div;
      if (src < 0 || src >= gather_limit) {
        if (lane == 0) report(status, kDevBadIndex);
        src = 0;
      }
    }
    const uint16_t *xr = x + src * cols;
    uint8_t *cr = codes + row * cols;
    for (int base = 0; base < cols; base += 256 * kRowUnroll) {
      uint4 v[kRowUnroll];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int col = base + u * 256 + lane * 8;
        v[u] = (col < cols) ? __ldcs(reinterpret_cast<const uint4 *>(xr + col)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int col = base + u * 256 + lane * 8;
        const uint32_t bm = absmax_bf16x2(absmax_bf16x2(v[u].x, v[u].y), absmax_bf16x2(v[u].z, v[u].w));
        uint32_t bmax = max(bm & 0x7FFFu, (bm >> 16) & 0x7FFFu);
        bmax = max(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 1));
        bmax = max(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, 2));
        const uint32_t code = mx_code<kCeil>(bmax);
        const float s = mx_inv_scale(code);
        uint2 out;
        out.x = e4m3x4_words(v[u].x, v[u].y, s);
        out.y = e4m3x4_words(v[u].z, v[u].w, s);
        if (col < cols) *reinterpret_cast<uint2 *>(cr + col) = out;
        const uint32_t pair = __byte_perm(code, __shfl_down_sync(0xFFFFFFFFu, code, 4), 0x0040);
        const uint32_t word = __byte_perm(pair, __shfl_down_sync(0xFFFFFFFFu, pair, 8), 0x5410);
        if ((lane & 15) == 0 && col < cols) {
          const int64_t cb = (base + u * 256) / 32 + lane / 4;
          *reinterpret_cast<uint32_t *>(sf + sf_offset(prow, cb, c4)) = word;
        }
      }
    }
  }
}

// ------------------------------------------------------------- column-wise --
// Tile = 128 padded positions (one 128-chunk of one group) x 128 columns.  The
// CTA stages the 128 x 128 bf16 tile in shared memory (rows past the group's end
// read as zeros; the next tile is already in registers), each thread quantizes
// one 32-block of two adjacent columns, the codes are staged transposed and
// leave as 128-byte rows, and the 128 x 4 scales of the tile are exactly one
// 512-byte tile of the scale layout.  A CTA walks tiles t = blockIdx.x, +gridDim.x,
// ... as (chunk, column block) pairs updated incrementally (no division), and
// the chunk's group only moves forward.
constexpr int kColTilePad = 8;  // bf16 elements of padding per staged row
constexpr int kColTileBytes = 128 * (128 + kColTilePad) * 2;
constexpr int kColOutBytes = 128 * (128 + 16);
constexpr int kColStageBytes = kColOutBytes + 512 + 512;  // codes, column scales, row scales of a tile
constexpr int kColSmemBytes = kColTileBytes + 2 * kColStageBytes;

// One tile of the walk: chunk j of the padded positions, column block cb, the
// chunk's group g, its first source row and how many of its 128 rows exist.
struct ColTile {
  int64_t j;
  int cb;
  int g;
  int valid;
  int64_t src0;
};

__device__ __forceinline__ void col_tile_locate(ColTile &t, const GroupTable &groups, int num_groups) {
  while (t.g + 1 < num_groups && groups.tiles[t.g + 1] <= t.j) ++t.g;
  const int64_t local0 = 128 * (t.j - groups.tiles[t.g]);
  const int64_t n_g = groups.off[t.g + 1] - groups.off[t.g];
  t.valid = static_cast<int>(n_g - local0 < 128 ? n_g - local0 : 128);
  t.src0 = groups.off[t.g] + local0;
}

// kMode kColsOnly: column-wise only.  kRowCol: also quantize the same tile
// row-wise (blocks of 32 along each row), so a tensor needed both ways is read
// once.  The tile's 128 padded positions are the row-wise scale layout's 128-row
// block j (both pad each group to 128 rows), so its row-wise scales are one
// 512-byte tile too.  kSwiGLUBwd: row-wise and column-wise, the tile produced from
// gate/up rows x = [g | u] (cols = 2 * inter) and dh [rows x inter]: tile column
// block jb covers gate columns 64 jb .. 64 jb + 63 (tile columns 0..63, dg) and
// the same up columns (tile columns 64..127, du), so g and dh are read once; the
// tile's halves land in different 128-column blocks of the outputs.
enum ColMode { kColsOnly = 0, kRowCol = 1, kSwiGLUBwd = 2 };

template <int kMode, bool kCeil>
__global__ void __launch_bounds__(256, 2) mxfp8_cols_kernel(const uint16_t *__restrict__ x, int64_t rows, int cols,
                                                         const int32_t *__restrict__ offsets, int num_groups,
                                                         uint8_t *__restrict__ codes_t, uint8_t *__restrict__ sf_t,
                                                         int64_t ld, int32_t *__restrict__ padded_offsets,
                                                         uint8_t *__restrict__ row_codes, uint8_t *__restrict__ row_sf,
                                                         int32_t *status, const uint16_t *__restrict__ dh,
                                                         uint16_t *__restrict__ d_out) {
  constexpr bool kRows = kMode != kColsOnly;
  constexpr bool kSw = kMode == kSwiGLUBwd;
  constexpr int kPre = kSw ? 12 : 8;  // 16-byte words of the next tile held per thread
  __shared__ GroupTable groups;
  __shared__ int ok_flag;
  extern __shared__ __align__(16) uint8_t col_smem[];
  auto tile = reinterpret_cast<uint16_t(*)[128 + kColTilePad]>(col_smem);
  // two staging buffers: tile t's outputs leave during tile t + 1, after its second
  // barrier, so that each tile needs two barriers instead of three
  auto outq_of = [&](int b) {
    return reinterpret_cast<uint8_t(*)[128 + 16]>(col_smem + kColTileBytes + b * kColStageBytes);
  };
  auto sfs_of = [&](int b) { return col_smem + kColTileBytes + b * kColStageBytes + kColOutBytes; };
  auto sfr_of = [&](int b) { return sfs_of(b) + 512; };  // row-wise scales of the tile (kRows)

  if (!load_groups(groups, offsets, num_groups, rows, &ok_flag)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, kDevBadOffsets);
    return;
  }
  const int tid = threadIdx.x;
  if (blockIdx.x == 0)
    for (int g = tid; g <= num_groups; g += blockDim.x) padded_offsets[g] = 128 * groups.tiles[g];

  const int64_t chunks = groups.tiles[num_groups];
  if (chunks * 128 > ld) {  // cannot happen for ld = fme_colwise_ld(); guards the stores
    if (blockIdx.x == 0 && tid == 0) report(status, kDevBadOffsets);
    return;
  }
  const int inter = cols / 2;  // kSwiGLUBwd only
  const int cblocks = kSw ? inter / 64 : cols / 128;
  const int64_t total = chunks * cblocks;
  const int64_t dj = gridDim.x / cblocks;
  const int dcb = gridDim.x % cblocks;
  auto advance = [&](ColTile &t) {
    t.j += dj;
    t.cb += dcb;
    if (t.cb >= cblocks) {
      t.cb -= cblocks;
      ++t.j;
    }
  };

  auto load_tile = [&](const ColTile &t, uint4 (&dst)[kPre]) {
    if constexpr (kSw) {
      // thread = (row pass * 32 + tid / 8, 8 consecutive gate columns): g, u, dh
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const int r = pass * 32 + (tid >> 3);
        const int c = t.cb * 64 + (tid & 7) * 8;
        const bool in = r < t.valid;
        const int64_t row = t.src0 + r;
        dst[3 * pass] = in ? __ldcs(reinterpret_cast<const uint4 *>(x + row * cols + c)) : make_uint4(0, 0, 0, 0);
        dst[3 * pass + 1] =
            in ? __ldcs(reinterpret_cast<const uint4 *>(x + row * cols + inter + c)) : make_uint4(0, 0, 0, 0);
        dst[3 * pass + 2] =
            in ? __ldcs(reinterpret_cast<const uint4 *>(dh + row * inter + c)) : make_uint4(0, 0, 0, 0);
      }
    } else {
#pragma unroll
      for (int pass = 0; pass < 8; ++pass) {
        const int r = pass * 16 + (tid >> 4);
        const int seg = tid & 15;
        dst[pass] = (r < t.valid)
                        ? __ldcs(reinterpret_cast<const uint4 *>(x + (t.src0 + r) * cols + t.cb * 128 + seg * 8))
                        : make_uint4(0, 0, 0, 0);
      }
    }
  };
  // Column-wise codes and scales (and kRows: row-wise scales) of tile pt, staged in
  // buffer b, to global memory.
  auto write_staged = [&](const ColTile &pt, int b) {
    const int cb = pt.cb;
    auto outq = outq_of(b);
    const uint8_t *sfs = sfs_of(b);
    const uint8_t *sfr = sfr_of(b);

#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int ch = pass * 32 + (tid >> 3);
      const int seg = tid & 7;
      const uint4 v = *reinterpret_cast<const uint4 *>(&outq[ch][seg * 16]);
      const int64_t gch = kSw ? (ch < 64 ? cb * 64 + ch : inter + cb * 64 + ch - 64) : static_cast<int64_t>(cb) * 128 + ch;
      *reinterpret_cast<uint4 *>(codes_t + gch * ld + pt.j * 128 + seg * 16) = v;
    }
    if constexpr (kSw) {
      // the gate and up halves are each half of a 512-byte scale tile: tile rows
      // (channels) 0..63 or 64..127 by the parity of cb (inter is a multiple of 128)
      const int odd = cb & 1;
      const int64_t t_g = cb / 2, t_u = (inter / 64 + cb) / 2;
      if (tid < 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(&sfs[tid * 16]);
        *reinterpret_cast<uint2 *>(sf_t + (t_g * (ld / 128) + pt.j) * 512 + tid * 16 + 8 * odd) = make_uint2(v.x, v.y);
        *reinterpret_cast<uint2 *>(sf_t + (t_u * (ld / 128) + pt.j) * 512 + tid * 16 + 8 * odd) = make_uint2(v.z, v.w);
      }
      {
        // row-wise scales: row r's 4-byte cell holds blocks (g0, g1, u0, u1)
        const int r = tid >> 1;
        const int half = tid & 1;
        const int cell = (r & 31) * 16 + (r >> 5) * 4;
        const uint16_t v = *reinterpret_cast<const uint16_t *>(&sfr[cell + 2 * half]);
        const int64_t tcol = half ? t_u : t_g;
        if (r < pt.valid)  // padding rows of the row-wise layout stay unwritten
          *reinterpret_cast<uint16_t *>(row_sf + (pt.j * (cols / 128) + tcol) * 512 + cell + 2 * odd) = v;
      }
    } else {
      if (tid < 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(&sfs[tid * 16]);
        *reinterpret_cast<uint4 *>(sf_t + (static_cast<int64_t>(cb) * (ld / 128) + pt.j) * 512 + tid * 16) = v;
      } else if (kRows && tid < 64) {
        // tile row i holds the row-wise scale words of rows i, i + 32, i + 64, i + 96;
        // padding rows (past the group's end) stay unwritten
        const int i = tid - 32;
        const uint4 v = *reinterpret_cast<const uint4 *>(&sfr[i * 16]);
        uint8_t *dst = row_sf + (pt.j * cblocks + cb) * 512 + i * 16;
        if (i + 96 < pt.valid) {
          *reinterpret_cast<uint4 *>(dst) = v;
        } else {
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (i + 32 * q < pt.valid) *reinterpret_cast<uint32_t *>(dst + 4 * q) = w[q];
        }
      }
    }
  };
  ColTile cur{static_cast<int64_t>(blockIdx.x) / cblocks, static_cast<int>(blockIdx.x % cblocks), 0, 0, 0};
  uint4 pre[kPre];
  if (cur.j < chunks) {
    col_tile_locate(cur, groups, num_groups);
    load_tile(cur, pre);
  }
  ColTile nxt = cur;
  advance(nxt);

  ColTile prev = cur;  // the tile whose outputs are staged in buffer buf ^ 1
  bool staged = false;
  int buf = 0;
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    const int cb = cur.cb;
    auto outq = outq_of(buf);
    uint8_t *sfs = sfs_of(buf);
    uint8_t *sfr = sfr_of(buf);
    __syncthreads();  // the tile buffer is free; the previous tile's staged outputs are complete
    if constexpr (kSw) {
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const int r = pass * 32 + (tid >> 3);
        const int c = (tid & 7) * 8;
        uint4 dg = make_uint4(0, 0, 0, 0), du = make_uint4(0, 0, 0, 0);
        if (r < cur.valid) swiglu_bwd_uint4(pre[3 * pass], pre[3 * pass + 1], pre[3 * pass + 2], dg, du);
        *reinterpret_cast<uint4 *>(&tile[r][c]) = dg;
        *reinterpret_cast<uint4 *>(&tile[r][64 + c]) = du;
      }
    } else {
#pragma unroll
      for (int pass = 0; pass < 8; ++pass)
        *reinterpret_cast<uint4 *>(&tile[pass * 16 + (tid >> 4)][(tid & 15) * 8]) = pre[pass];
      if constexpr (kRows) {
        // the row-wise pass from the registers the tile came in: the four lanes of a
        // row's 32-block (8 values each) take its amax with two shuffles, and each
        // lane writes its 8 codes (a warp: two full 128-byte rows).  Measured against
        // the pass re-reading the staged tile: 1.371-1.434 -> 1.320 ms for the
        // 262144 x 7168 row + column quantization, outputs bit-identical.
        const int seg = tid & 15;
#pragma unroll
        for (int pass = 0; pass < 8; ++pass) {
          const int r = pass * 16 + (tid >> 4);
          const uint4 v = pre[pass];
          uint32_t m = absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w));
          m = absmax_bf16x2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
          m = absmax_bf16x2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
          const uint32_t code = mx_code<kCeil>(max(m & 0x7FFFu, (m >> 16) & 0x7FFFu));
          const float sc = mx_inv_scale(code);
          const uint2 wv = make_uint2(e4m3x4_words(v.x, v.y, sc), e4m3x4_words(v.z, v.w, sc));
          if (r < cur.valid)  // rows past the group's end are not stored
            *reinterpret_cast<uint2 *>(row_codes + (cur.src0 + r) * cols + cb * 128 + seg * 8) = wv;
          if ((seg & 3) == 0) sfr[(r & 31) * 16 + (r >> 5) * 4 + (seg >> 2)] = static_cast<uint8_t>(code);
        }
      }
    }
    __syncthreads();
    if (staged) write_staged(prev, buf ^ 1);
    if (nxt.j < chunks) {
      col_tile_locate(nxt, groups, num_groups);
      load_tile(nxt, pre);
      // the tile after next: one 128-byte line per thread into L2, so that its
      // register loads a tile from now find it there
      ColTile nn = nxt;
      advance(nn);
      if (nn.j < chunks) {
        col_tile_locate(nn, groups, num_groups);
        const int r = tid & 127;
        if (r < nn.valid) {
          const int64_t row = nn.src0 + r;
          const uint16_t *line;
          if constexpr (kSw) {
            line = (tid < 128) ? x + row * cols + nn.cb * 64 : x + row * cols + inter + nn.cb * 64;
          } else {
            line = x + row * cols + nn.cb * 128 + (tid >> 7) * 64;
          }
          asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
          if constexpr (kSw) {
            if (tid < 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(dh + row * inter + nn.cb * 64));
          }
        }
      }
    }

    // thread = (channel pair cp, 32-position block b): both channels' 32 values
    // come in with one 32-bit shared load per position
    {
      const int cp = tid & 63;
      const int b = tid >> 6;
      uint32_t vals[32];
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        vals[i] = *reinterpret_cast<const uint32_t *>(&tile[32 * b + i][2 * cp]);
        m = absmax_bf16x2(m, vals[i]);
      }
      const uint32_t code_lo = mx_code<kCeil>(m & 0x7FFFu);
      const uint32_t code_hi = mx_code<kCeil>((m >> 16) & 0x7FFFu);
      const float s_lo = mx_inv_scale(code_lo);
      const float s_hi = mx_inv_scale(code_hi);
      uint32_t wl[8], wh[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t *v = vals + 4 * q;
        wl[q] = e4m3x4_scaled(v[0] << 16, v[1] << 16, v[2] << 16, v[3] << 16, s_lo);
        wh[q] = e4m3x4_scaled(v[0] & 0xFFFF0000u, v[1] & 0xFFFF0000u, v[2] & 0xFFFF0000u, v[3] & 0xFFFF0000u, s_hi);
      }
      const int c = 2 * cp;
      *reinterpret_cast<uint4 *>(&outq[c][32 * b]) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      *reinterpret_cast<uint4 *>(&outq[c][32 * b + 16]) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
      *reinterpret_cast<uint4 *>(&outq[c + 1][32 * b]) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
      *reinterpret_cast<uint4 *>(&outq[c + 1][32 * b + 16]) = make_uint4(wh[4], wh[5], wh[6], wh[7]);
      sfs[(c & 31) * 16 + (c >> 5) * 4 + b] = static_cast<uint8_t>(code_lo);
      sfs[((c + 1) & 31) * 16 + ((c + 1) >> 5) * 4 + b] = static_cast<uint8_t>(code_hi);
    }
    if (kSw) {
      // the SwiGLU backward's row-wise pass, from the staged d(gate/up) tile:
      // thread = (row r, 32-column block b) for 2 of the tile's 512 pairs; a
      // quarter-warp takes 8 consecutive rows of one block (conflict-free 16-byte
      // reads); rows past the group's end are not stored
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int p = tid + 256 * h;
        const int b = (p >> 3) & 3;
        const int r = (p & 7) + 8 * (p >> 5);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = *reinterpret_cast<const uint4 *>(&tile[r][32 * b + 8 * i]);
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 16; i += 2) m = absmax_bf16x2(m, absmax_bf16x2(w[i], w[i + 1]));
        const uint32_t code = mx_code<kCeil>(max(m & 0x7FFFu, (m >> 16) & 0x7FFFu));
        const float s = mx_inv_scale(code);
        uint32_t words[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) words[q] = e4m3x4_words(w[2 * q], w[2 * q + 1], s);
        if (r < cur.valid) {
          const int col = b < 2 ? cb * 64 + 32 * b : inter + cb * 64 + 32 * (b - 2);
          uint4 *dst = reinterpret_cast<uint4 *>(row_codes + (cur.src0 + r) * cols + col);
          dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
          dst[1] = make_uint4(words[4], words[5], words[6], words[7]);
        }
        sfr[(r & 31) * 16 + (r >> 5) * 4 + b] = static_cast<uint8_t>(code);
      }
    }
    if constexpr (kSw) {
      if (d_out != nullptr) {
#pragma unroll
        for (int pass = 0; pass < 8; ++pass) {
          const int r = pass * 16 + (tid >> 4);
          const int seg = tid & 15;
          if (r < cur.valid) {
            const uint4 v = *reinterpret_cast<const uint4 *>(&tile[r][seg * 8]);
            const int col = seg < 8 ? cb * 64 + seg * 8 : inter + cb * 64 + (seg - 8) * 8;
            *reinterpret_cast<uint4 *>(d_out + (cur.src0 + r) * cols + col) = v;
          }
        }
      }
    }
    prev = cur;
    staged = true;
    buf ^= 1;
    cur = nxt;
    advance(nxt);
  }
  __syncthreads();
  if (staged) write_staged(prev, buf ^ 1);
}

cudaError_t launch_quantize_mxfp8_rows(const LaunchMxfp8 &a) {
  const int threads = 256;
  const int64_t need = (a.rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 8;
  const int blocks = static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
  auto kernel = a.ceil_scale ? mxfp8_rows_kernel<true> : mxfp8_rows_kernel<false>;
  kernel<<<blocks, threads, 0, a.stream>>>(static_cast<const uint16_t *>(a.x), a.rows, static_cast<int>(a.cols),
                                           a.offsets, a.num_groups, a.codes, a.sf, a.status, a.gather,
                                           a.gather_div, a.gather_limit);
  return cudaGetLastError();
}

template <int kMode, bool kCeil = false>
static cudaError_t launch_cols(const LaunchMxfp8 &a, uint8_t *row_codes, uint8_t *row_sf) {
  const int threads = 256;
  const int64_t tiles = (a.ld / 128) * (a.cols / 128);  // kSwiGLUBwd: inter / 64 = cols / 128 column blocks
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 2;
  const int blocks = static_cast<int>(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
  auto kernel = mxfp8_cols_kernel<kMode, kCeil>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kColSmemBytes);
  if (err != cudaSuccess) return err;
  kernel<<<blocks, threads, kColSmemBytes, a.stream>>>(
      static_cast<const uint16_t *>(a.x), a.rows, static_cast<int>(a.cols), a.offsets, a.num_groups, a.codes, a.sf,
      a.ld, a.padded_offsets, row_codes, row_sf, a.status, static_cast<const uint16_t *>(a.dh),
      static_cast<uint16_t *>(a.d_out));
  return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8_cols(const LaunchMxfp8 &a) {
  return a.ceil_scale ? launch_cols<kColsOnly, true>(a, nullptr, nullptr)
                      : launch_cols<kColsOnly, false>(a, nullptr, nullptr);
}

cudaError_t launch_quantize_mxfp8_rowcol(const LaunchMxfp8 &a, uint8_t *row_codes, uint8_t *row_sf) {
  return launch_cols<kRowCol>(a, row_codes, row_sf);
}

cudaError_t launch_swiglu_bwd_mxfp8(const LaunchMxfp8 &a, uint8_t *row_codes, uint8_t *row_sf) {
  return launch_cols<kSwiGLUBwd>(a, row_codes, row_sf);
}

}  // namespace fme

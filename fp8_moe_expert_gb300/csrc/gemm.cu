// gemm.cu -- block-scaled grouped GEMMs on the tcgen05 tensor cores, CTA pairs.
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1: the MoE
// layer's grouped GEMMs run as block-scaled tensor-core MMAs on Blackwell (the
// scales are applied inside the systolic-array multiply); NVFP4 with a per-token
// FP32 scale applied in the GEMM epilogue for the forward, MXFP8 for the
// backward.  "Scaling and Optimizing Frontier Model Training", "MXFP8 expert
// kernels": grouped GEMMs over the experts' routed tokens.
//
// One persistent kernel per call.  CTAs run in pairs (a cluster of 2 on two
// SMs); a pair computes 256 x 256 output tiles with cta_group::2 MMAs (M = 256:
// 128 rows in each CTA's tensor memory).  Each CTA stages its own 128 rows of A
// and its half (128 rows) of the tile's 256 B rows, so a pair moves 1.5x fewer
// operand bytes per flop than a single CTA with a 128 x 256 tile, and each
// scale copy into tensor memory serves twice the MMA work.  The forward's B
// scales arrive pre-replicated (quantize_nvfp4_weights), so B needs one wide
// tensor-memory copy per 64-deep step instead of two narrow ones.  12 warps per CTA:
//   warp 0      TMA producer (both CTAs): A, B and their scale tiles into a
//               4-6 stage ring; every copy of the pair completes on a barrier of
//               the leader CTA, the scale tiles (issued first) on "sf_landed",
//               A and B on "full", so that the scale copies below overlap the
//               operand loads instead of following them;
//   warp 1      allocates 512 tensor-memory columns in both CTAs together; in the
//               leader, one thread issues the block-scaled MMAs (kind::mxf4nvf4
//               or kind::mxf8f6f4, M = 256, N = 256); commits free the stage in
//               both CTAs and, at the end of a tile, fill both CTAs' accumulators;
//   warps 10-11 in the leader, one thread of each copies half of each stage's
//               scale tiles into a ring of 4 tensor-memory buffers (tcgen05.cp)
//               ahead of the MMAs (one issuing thread cannot keep up with the
//               FP4 MMAs: each copy occupies it for about 90 cycles);
//   warps 2-9   epilogue (both CTAs): tcgen05.ld its own 128 x 256 fp32
//               accumulator (each warp a 32-lane quarter and half the columns)
//               into registers, release it to the leader, then apply the
//               per-token and per-column FP32 scales (forward), round to bf16,
//               and transpose each 32 x 32 block through shared memory so that a
//               store instruction writes 64 contiguous bytes of each of 8 rows
//               (rows past the expert's last row are skipped), overlapping the
//               next tile's MMAs.
// Kinds: the NVFP4 forward (kind::mxf4nvf4, per-token and per-column FP32 scales
// in the epilogue), the MXFP8 forward (kind::mxf8f6f4, same operand layout), dgrad
// and wgrad (kind::mxf8f6f4).
// Both CTAs walk the same tile sequence, derived in shared memory from the
// per-expert offsets: forward and dgrad go expert by expert, 256-row blocks of
// each expert's rows, 256-column blocks fastest; wgrad goes expert by expert in
// decreasing order of work (largest contraction first) and writes zeros for
// experts without rows.  There is no split over K: each output element is one
// accumulation, so a row's result does not depend on other rows.
#include "fme_device.cuh"
#include "fme_launch.h"

namespace fme {

constexpr int kBM = 128;           // rows per CTA
constexpr int kPairM = 256;        // rows per pair tile
constexpr int kBN = 256;           // columns per tile
constexpr int kHalfN = kBN / 2;    // B rows staged by each CTA
constexpr int kStageKBytes = 128;  // bytes of K per row per stage (one swizzle row)
constexpr int kThreads = 384;      // producer, MMA, 8 epilogue warps, 2 scale copiers
constexpr int kCopierWarp = 10;    // and 11
constexpr int kCopiers = 2;
constexpr int kSfBuffers = 4;      // tensor-memory scale buffers between the copier and the MMA issuer
constexpr int kMaxStages = 6;
constexpr int kOutBoxBytes = 32 * 32 * 2;            // one 32-row x 32-column bf16 block
constexpr int kSwBytes = 128 * 4;                    // a warp's 128 column scales (forward)
constexpr int kOutBytes = 8 * (kOutBoxBytes + kSwBytes);  // staging block + column scales per epilogue warp
constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = kBM * kStageKBytes;
constexpr int kBBytes = kHalfN * kStageKBytes;
constexpr int kAccEmptyArrivals = 2 * 8;  // one per epilogue warp of the pair

template <GemmKind K>
struct Cfg {
  static constexpr bool kFp4 = (K == GemmKind::kFwdNvfp4);
  static constexpr int kKPerStage = kFp4 ? 256 : 128;  // elements of K per stage
  static constexpr int kAtoms = kFp4 ? 4 : 1;          // 512-byte scale tiles per 128 rows per stage
  static constexpr int kSfaBytes = 512 * kAtoms;       // this CTA's 128 rows
  // All 256 B rows of the tile.  FP4: the weights' replicated layout, 4096 bytes per
  // 64-deep step (the two 512-byte tiles four times each, one wide copy); FP8: the
  // plain tiles (two 512-byte tiles per step).
  static constexpr int kSfbBytes = kFp4 ? 4096 * kAtoms : 2 * 512 * kAtoms;
  static constexpr int kSfaCols = 4 * kAtoms;          // tensor-memory columns per stage
  static constexpr int kSfbCols = 8 * kAtoms;
  static constexpr int kSfCols = kSfaCols + kSfbCols;
  static constexpr int kStages = kFp4 ? 5 : 6;  // ring depth when the shared memory allows
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  // Both CTAs' copies land on the leader's barriers: the operands on "full", the
  // scale tiles (issued first) on "sf_landed".
  static constexpr int kOperandTx = 2 * (kABytes + kBBytes);
  static constexpr int kScaleTx = 2 * (kSfaBytes + kSfbBytes);
  static_assert(kStages <= kMaxStages, "stage count");
  static_assert(kBN + kSfBuffers * kSfCols <= static_cast<int>(kTmemCols), "tensor memory budget");
};

struct SharedState {
  uint64_t full[kMaxStages];       // the stage's A and B tiles have landed
  uint64_t sf_landed[kMaxStages];  // the stage's scale tiles have landed
  uint64_t empty[kMaxStages];
  uint64_t sf_full[kSfBuffers];   // scales of a stage are in tensor-memory buffer b (one arrival per copier)
  uint64_t sf_empty[kSfBuffers];  // the MMAs reading buffer b are done
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint64_t drain_cp[kCopiers];
  uint32_t tmem_base;
  int abort_flag;
  int ok_flag;
};

// Group tables (G + 1 entries each) in dynamic shared memory, after the operand
// ring and the output staging boxes.
struct Groups {
  int32_t *off;    // fwd, dgrad: row offsets;           wgrad: padded offsets
  int32_t *tiles;  // fwd, dgrad: 128-row tile prefix;   wgrad: experts by decreasing work
  int32_t *pair;   // fwd, dgrad: 256-row tile prefix
};

// Dynamic shared memory: [operand ring][output staging][group tables], with
// 1024 bytes of slack to align the ring for the 128-byte swizzle.
__host__ __device__ __forceinline__ int64_t ring_bytes(int stages, int stage_bytes) {
  return (static_cast<int64_t>(stages) * stage_bytes + 1023) / 1024 * 1024;
}
__host__ __device__ __forceinline__ int64_t gemm_smem_bytes(int stages, int stage_bytes, int num_groups) {
  return 1024 + ring_bytes(stages, stage_bytes) + kOutBytes + 12 * static_cast<int64_t>(num_groups + 1);
}

struct Tile {
  int32_t e;
  int32_t num_k;           // K stages; 0 = expert without rows (wgrad): output zeros
  int32_t rows_valid;      // rows of this CTA's 128 that belong to the expert (may be <= 0)
  int64_t y_off;           // element offset of this CTA's first output element
  int32_t a_y, b_y;        // TMA row coordinates of this CTA's A rows and B half
  int32_t a_x0, b_x0;      // TMA K coordinates (bytes) of the first stage
  int32_t sfa_row;         // 128-row scale block of this CTA's A rows
  int32_t sfb_row;         // FP8: first of the two 128-row scale blocks of the tile's B rows;
                           // FP4: first 2 KB row of the tile's replicated scale blocks
  int32_t sfa_x0, sfb_x0;  // 512-byte scale tile index of the first stage
  int32_t n0;              // first output column
};

template <GemmKind K>
__device__ __forceinline__ int64_t total_tiles(const LaunchGemm &p, const Groups &g) {
  const int64_t nb = p.n / kBN;
  if (K == GemmKind::kWgradMxfp8) return static_cast<int64_t>(p.num_experts) * (p.m / kPairM) * nb;
  return static_cast<int64_t>(g.pair[p.num_experts]) * nb;
}

template <GemmKind K>
__device__ __forceinline__ Tile tile_at(const LaunchGemm &p, const Groups &s, int64_t t, int rank) {
  using C = Cfg<K>;
  Tile tl;
  const int64_t nb_count = p.n / kBN;
  if (K == GemmKind::kWgradMxfp8) {
    const int64_t mb_count = p.m / kPairM;
    const int64_t per = mb_count * nb_count;
    const int order = static_cast<int>(t / per);
    const int64_t rem = t % per;
    const int64_t mb = rem / nb_count;
    const int64_t nb = rem % nb_count;
    const int e = s.tiles[order];
    const int32_t p0 = s.off[e];
    const int64_t row0 = mb * kPairM + rank * kBM;
    tl.e = e;
    tl.num_k = (s.off[e + 1] - p0) / 128;
    tl.rows_valid = kBM;
    tl.n0 = static_cast<int32_t>(nb * kBN);
    tl.y_off = (static_cast<int64_t>(e) * p.m + row0) * p.n + nb * kBN;
    tl.a_y = static_cast<int32_t>(row0);
    tl.b_y = static_cast<int32_t>(nb * kBN + rank * kHalfN);
    tl.a_x0 = p0;
    tl.b_x0 = p0;
    tl.sfa_row = static_cast<int32_t>(row0 / 128);
    tl.sfb_row = static_cast<int32_t>(2 * nb);
    tl.sfa_x0 = p0 / 128;
    tl.sfb_x0 = p0 / 128;
  } else {
    const int64_t g = t / nb_count;
    const int64_t nb = t % nb_count;
    const int e = find_group(s.pair, p.num_experts, g);
    const int64_t mb = 2 * (g - s.pair[e]) + rank;  // this CTA's 128-row block within the expert
    const int64_t r0 = s.off[e] + mb * kBM;
    const int64_t n_e = s.off[e + 1] - s.off[e];
    const int64_t left = n_e - mb * kBM;
    tl.e = e;
    tl.num_k = static_cast<int32_t>(p.k / C::kKPerStage);
    tl.rows_valid = static_cast<int32_t>(left < kBM ? left : kBM);
    tl.n0 = static_cast<int32_t>(nb * kBN);
    tl.y_off = r0 * p.n + nb * kBN;
    tl.a_y = static_cast<int32_t>(r0);
    tl.a_x0 = 0;
    tl.sfa_row = s.tiles[e] + static_cast<int32_t>(mb);
    tl.sfa_x0 = 0;
    if (K == GemmKind::kFwdNvfp4 || K == GemmKind::kFwdMxfp8) {
      // B = stacked weights, expert e's rows e*n .. e*n+n-1, K contiguous
      const int64_t brow = static_cast<int64_t>(e) * p.n + nb * kBN;
      tl.b_y = static_cast<int32_t>(brow + rank * kHalfN);
      tl.b_x0 = 0;
      tl.sfb_row = (K == GemmKind::kFwdNvfp4) ? static_cast<int32_t>((brow / kBN) * (p.k / 64) * 2)
                                               : static_cast<int32_t>(brow / 128);
      tl.sfb_x0 = 0;
    } else {
      tl.b_y = static_cast<int32_t>(nb * kBN + rank * kHalfN);
      tl.b_x0 = static_cast<int32_t>(static_cast<int64_t>(e) * p.k);
      tl.sfb_row = static_cast<int32_t>(2 * nb);
      tl.sfb_x0 = static_cast<int32_t>(static_cast<int64_t>(e) * p.k / 128);
    }
  }
  return tl;
}

// Build the tile tables (the same in both CTAs of a pair); returns false in
// every thread for malformed offsets.
template <GemmKind K>
__device__ bool prepare(const LaunchGemm &p, SharedState &s, const Groups &g) {
  if (K != GemmKind::kWgradMxfp8) {
    if (!load_groups(g.off, g.tiles, p.offsets, p.num_experts, p.m, &s.ok_flag)) return false;
    if (threadIdx.x == 0) {
      int32_t acc = 0;
      for (int e = 0; e < p.num_experts; ++e) {
        g.pair[e] = acc;
        acc += (g.off[e + 1] - g.off[e] + kPairM - 1) / kPairM;
      }
      g.pair[p.num_experts] = acc;
    }
    __syncthreads();
    return true;
  }
  // wgrad: padded offsets, multiples of 128, rising from 0 within both operands
  if (threadIdx.x == 0) {
    bool ok = true;
    int32_t prev = 0;
    for (int e = 0; e <= p.num_experts; ++e) {
      const int32_t v = __ldg(p.offsets + e);
      if ((e == 0 && v != 0) || v < prev || (v & 127) != 0) ok = false;
      g.off[e] = v;
      prev = v;
    }
    if (prev > p.lda || prev > p.ldb) ok = false;
    s.ok_flag = ok ? 1 : 0;
  }
  __syncthreads();
  if (!s.ok_flag) return false;
  for (int e = threadIdx.x; e < p.num_experts; e += blockDim.x) {
    const int32_t w = g.off[e + 1] - g.off[e];
    int rank = 0;
    for (int f = 0; f < p.num_experts; ++f) {
      const int32_t wf = g.off[f + 1] - g.off[f];
      rank += (wf > w) || (wf == w && f < e);
    }
    g.tiles[rank] = e;
  }
  __syncthreads();
  return true;
}

// Scale (forward: (acc * S_x[t]) * S_w[n], fp32, two values per packed f32x2
// multiply) and round to bf16 32 consecutive outputs of one row, two per word.
// `sw` (forward) points at the 32 column scales in shared memory; every lane
// reads the same addresses (broadcast).
template <GemmKind K>
__device__ __forceinline__ void convert_chunk(uint32_t (&packed)[16], const uint32_t (&v)[32], float sa,
                                              const float *sw) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float2 f0 = make_float2(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]));
    float2 f1 = make_float2(__uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
    if (K == GemmKind::kFwdNvfp4) {
      const float4 b = *reinterpret_cast<const float4 *>(sw + 4 * j);
      f0 = __fmul2_rn(__fmul2_rn(f0, make_float2(sa, sa)), make_float2(b.x, b.y));
      f1 = __fmul2_rn(__fmul2_rn(f1, make_float2(sa, sa)), make_float2(b.z, b.w));
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(f0.x, f0.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(f1.x, f1.y);
    packed[2 * j] = *reinterpret_cast<const uint32_t *>(&lo);
    packed[2 * j + 1] = *reinterpret_cast<const uint32_t *>(&hi);
  }
}

// A 32 x 32 block of bf16 outputs (row `lane` of the warp's 32 rows in
// `packed`) to global memory through the warp's 2 KB staging block: row r's
// 16-byte chunk j goes to chunk j ^ ((r >> 1) & 3) of its 64-byte staging row
// (conflict-free writes and reads), then lane l writes chunk l % 4 of row
// 8 i + l / 4 for i = 0..3: each store instruction covers 64 contiguous bytes of
// 8 rows.  Rows at or past `rows_valid` are not written.
__device__ __forceinline__ void store_block(__nv_bfloat16 *dst, int64_t ld, int rows_valid, uint8_t *stage,
                                            int lane, const uint32_t (&packed)[16]) {
  {
    uint8_t *row = stage + lane * 64;
    const int x = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4 *>(row + 16 * (j ^ x)) =
          make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
  }
  __syncwarp();
  const int j = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    const uint4 v = *reinterpret_cast<const uint4 *>(stage + r * 64 + 16 * (j ^ ((r >> 1) & 3)));
    if (r < rows_valid) *reinterpret_cast<uint4 *>(dst + r * ld + 8 * j) = v;
  }
  __syncwarp();
}

template <GemmKind K>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ LaunchGemm p) {
  using C = Cfg<K>;
  __shared__ SharedState s;
  extern __shared__ uint8_t dyn_smem[];
  const int S = p.stages;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t *smem_a = smem;
  uint8_t *smem_b = smem_a + S * kABytes;
  uint8_t *smem_sfa = smem_b + S * kBBytes;
  uint8_t *smem_sfb = smem_sfa + S * C::kSfaBytes;
  uint8_t *smem_out = smem + ring_bytes(S, C::kStageBytes);
  int32_t *gmem = reinterpret_cast<int32_t *>(smem_out + kOutBytes);
  const Groups grp{gmem, gmem + (p.num_experts + 1), gmem + 2 * (p.num_experts + 1)};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(pair::cta_rank());
  const int64_t pair_id = blockIdx.x >> 1;
  const int64_t pairs = gridDim.x >> 1;

  // Both CTAs of a pair see the same offsets, so both return here or neither does.
  if (!prepare<K>(p, s, grp)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.status, kDevBadOffsets);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.sf_landed[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < kSfBuffers; ++i) {
      mbar_init(&s.sf_full[i], kCopiers);
      mbar_init(&s.sf_empty[i], 1);
    }
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, kAccEmptyArrivals);
    mbar_init(&s.drain, 1);
    for (int i = 0; i < kCopiers; ++i) mbar_init(&s.drain_cp[i], 1);
    s.abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
    prefetch_tensormap(&p.map_a);
    prefetch_tensormap(&p.map_b);
    prefetch_tensormap(&p.map_sfa);
    prefetch_tensormap(&p.map_sfb);
  }
  if (warp == 1) {
    pair::tmem_alloc(&s.tmem_base, kTmemCols);
    pair::tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  pair::cluster_sync();  // both CTAs' barriers exist before any copy or arrive crosses the pair
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int *abort_flag = &s.abort_flag;
  const int64_t total = total_tiles<K>(p, grp);

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- producer
    uint32_t stage = 0, phase = 0;
    for (int64_t t = pair_id; t < total; t += pairs) {
      const Tile tl = tile_at<K>(p, grp, t, rank);
      bool stop = false;
      for (int ks = 0; ks < tl.num_k; ++ks) {
        if (!mbar_wait(&s.empty[stage], phase ^ 1, abort_flag, p.status)) {
          stop = true;
          break;
        }
        // Scales first, on their own barrier: the copiers start on them while the
        // operands are still arriving, so the tensor-memory copies are done by the
        // time the MMAs could start (the copy latency was on the critical path).
        if (rank == 0) mbar_arrive_expect_tx(&s.sf_landed[stage], C::kScaleTx);
        const uint32_t sbar = pair::map_to_rank(&s.sf_landed[stage], 0);
        pair::tma_load_2d(smem_sfa + stage * C::kSfaBytes, &p.map_sfa, sbar, (tl.sfa_x0 + ks * C::kAtoms) * 64,
                          tl.sfa_row);
        if (C::kFp4)  // four 64-deep steps of replicated blocks: 8 rows of 2 KB
          pair::tma_load_2d(smem_sfb + stage * C::kSfbBytes, &p.map_sfb, sbar, 0, tl.sfb_row + 8 * ks);
        else
          pair::tma_load_2d(smem_sfb + stage * C::kSfbBytes, &p.map_sfb, sbar, (tl.sfb_x0 + ks * C::kAtoms) * 64,
                            tl.sfb_row);
        if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], C::kOperandTx);
        const uint32_t bar = pair::map_to_rank(&s.full[stage], 0);
        pair::tma_load_2d(smem_a + stage * kABytes, &p.map_a, bar, tl.a_x0 + ks * kStageKBytes, tl.a_y);
        pair::tma_load_2d(smem_b + stage * kBBytes, &p.map_b, bar, tl.b_x0 + ks * kStageKBytes, tl.b_y);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (stop) break;
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------ MMA issuer (leader)
    uint32_t stage = 0, phase = 0, acc_phase = 0, buf = 0, buf_phase = 0;
    bool stop = false;
    const uint32_t sf_base = tmem + kBN;
    for (int64_t t = pair_id; t < total && !stop; t += pairs) {
      const Tile tl = tile_at<K>(p, grp, t, 0);
      if (tl.num_k == 0) continue;
      if (!mbar_wait(&s.acc_empty, acc_phase ^ 1, abort_flag, p.status)) break;
      tc_fence_after();
      for (int ks = 0; ks < tl.num_k; ++ks) {
        if (!mbar_wait(&s.full[stage], phase, abort_flag, p.status) ||
            !mbar_wait(&s.sf_full[buf], buf_phase, abort_flag, p.status)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = sf_base + buf * C::kSfCols;
        const uint32_t sfb_t = sfa_t + C::kSfaCols;
        const uint32_t a_s = smem_u32(smem_a + stage * kABytes);
        const uint32_t b_s = smem_u32(smem_b + stage * kBBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = desc_sw128_kmajor(a_s + kk * 32);
          const uint64_t bd = desc_sw128_kmajor(b_s + kk * 32);
          const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
          if (C::kFp4)
            pair::mma_nvf4(tmem, ad, bd, pair::idesc_nvf4(kBN), sfa_t + 4 * kk, sfb_t + 8 * kk, acc);
          else
            pair::mma_mxf8(tmem, ad, bd, pair::idesc_mxf8(kBN, kk), sfa_t, sfb_t, acc);
        }
        pair::commit_both(&s.empty[stage]);
        pair::commit_local(&s.sf_empty[buf]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
        if (++buf == kSfBuffers) {
          buf = 0;
          buf_phase ^= 1;
        }
      }
      if (stop) break;
      pair::commit_both(&s.acc_full);
      acc_phase ^= 1;
    }
    // every tensor-core operation of the pair has finished before memory is released
    pair::commit_local(&s.drain);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&s.drain, 0) && globaltimer() - t0 < kWaitLimitNs / 4) {
    }
  } else if (warp >= kCopierWarp && warp < kCopierWarp + kCopiers && lane == 0 && rank == 0) {
    // --------------------------------------------------- scale copiers (leader)
    // Copy each stage's scale tiles (both CTAs, tcgen05.cp.cta_group::2) into the
    // next free tensor-memory buffer while the MMA issuer works on earlier stages,
    // then arrive on the buffer's "full" barrier.  FP4: copier 0 takes A (one
    // 32x128b.warpx4 per 64-deep step), copier 1 takes B (one 128x256b copy of the
    // replicated block per step: each copy costs the tensor core about the same
    // whatever its size, so one wide copy beats two narrow ones).  FP8: the stage's
    // three copies, A, B-low, B-high, alternate between the copiers.
    const int who = warp - kCopierWarp;
    uint32_t stage = 0, phase = 0, buf = 0, buf_phase = 0;
    bool stop = false;
    const uint32_t sf_base = tmem + kBN;
    for (int64_t t = pair_id; t < total && !stop; t += pairs) {
      const Tile tl = tile_at<K>(p, grp, t, 0);
      for (int ks = 0; ks < tl.num_k; ++ks) {
        if (!mbar_wait(&s.sf_landed[stage], phase, abort_flag, p.status) ||
            !mbar_wait(&s.sf_empty[buf], buf_phase ^ 1, abort_flag, p.status)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = sf_base + buf * C::kSfCols;
        const uint32_t sfb_t = sfa_t + C::kSfaCols;
        const uint32_t sfa_s = smem_u32(smem_sfa + stage * C::kSfaBytes);
        const uint32_t sfb_s = smem_u32(smem_sfb + stage * C::kSfbBytes);
        if (C::kFp4) {
#pragma unroll
          for (int i = 0; i < C::kAtoms; ++i) {
            if (who == 0)
              pair::copy_scales(sfa_t + 4 * i, desc_scale_tile(sfa_s + 512 * i));
            else
              pair::copy_scales_wide(sfb_t + 8 * i, desc_scale_rep(sfb_s + 4096 * i));
          }
        } else {
#pragma unroll
          for (int i = 0; i < C::kAtoms; ++i) {
            if ((3 * i) % kCopiers == who) pair::copy_scales(sfa_t + 4 * i, desc_scale_tile(sfa_s + 512 * i));
            if ((3 * i + 1) % kCopiers == who) pair::copy_scales(sfb_t + 8 * i, desc_scale_tile(sfb_s + 512 * i));
            if ((3 * i + 2) % kCopiers == who)
              pair::copy_scales(sfb_t + 8 * i + 4, desc_scale_tile(sfb_s + C::kSfbBytes / 2 + 512 * i));
          }
        }
        pair::commit_local(&s.sf_full[buf]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
        if (++buf == kSfBuffers) {
          buf = 0;
          buf_phase ^= 1;
        }
      }
    }
    pair::commit_local(&s.drain_cp[who]);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&s.drain_cp[who], 0) && globaltimer() - t0 < kWaitLimitNs / 4) {
    }
  } else if (warp >= 2 && warp < kCopierWarp) {
    // --------------------------------------------------------------- epilogue
    // Warp w reads tensor-memory lane quarter w % 4 (rows 32(w%4) .. +31) and
    // column half (w - 2) / 4.  All 128 accumulator columns of a thread are
    // loaded before the accumulator is released to the leader.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const int c0 = half * (kBN / 2);
    const uint32_t leader_acc_empty = pair::map_to_rank(&s.acc_empty, 0);
    uint8_t *stage_blk = smem_out + (warp - 2) * kOutBoxBytes;
    float *sw = reinterpret_cast<float *>(smem_out + 8 * kOutBoxBytes + (warp - 2) * kSwBytes);
    uint32_t acc_phase = 0;
    __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(p.y);
    for (int64_t t = pair_id; t < total; t += pairs) {
      const Tile tl = tile_at<K>(p, grp, t, rank);
      const bool valid = r < tl.rows_valid;
      __nv_bfloat16 *yrow = y + tl.y_off + static_cast<int64_t>(r) * p.n + c0;
      const bool acc_out = K == GemmKind::kWgradMxfp8 && p.accumulate;
      if (tl.num_k == 0) {  // an empty expert: dW = 0 (accumulating: nothing to add)
        if (valid && !acc_out)
          for (int c = 0; c < kBN / 2; c += 8) *reinterpret_cast<uint4 *>(yrow + c) = make_uint4(0, 0, 0, 0);
        continue;
      }
      // the forward's scales of this warp's rows and columns, fetched while the MMAs run
      float sa = 1.0f;
      float4 swv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (K == GemmKind::kFwdNvfp4) {
        if (valid) sa = __ldg(p.a_scale + tl.a_y + r);
        swv = __ldg(reinterpret_cast<const float4 *>(p.b_scale + static_cast<int64_t>(tl.e) * p.n + tl.n0 + c0) +
                    lane);
      }
      if (!mbar_wait(&s.acc_full, acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      uint32_t v0[32], v1[32], v2[32], v3[32];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + c0;
      tmem_ld_32x32(taddr, v0);
      tmem_ld_32x32(taddr + 32, v1);
      tmem_ld_32x32(taddr + 64, v2);
      tmem_ld_32x32(taddr + 96, v3);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) pair::arrive_remote_relaxed(leader_acc_empty);  // registers hold the data
      acc_phase ^= 1;
      if (K == GemmKind::kFwdNvfp4) {
        reinterpret_cast<float4 *>(sw)[lane] = swv;
        __syncwarp();
      }
      if (acc_out) {
        // fp32 gradient accumulation, one unfused add per element (each element has
        // one owner).  Each 32 x 16 fp32 half-chunk goes through the warp's 2 KB
        // staging block (16-byte chunk j of row r at j ^ ((r >> 1) & 3)), so that
        // four lanes read-add-write 64 contiguous bytes of one row and an
        // instruction covers 8 rows.
        float *ywarp = static_cast<float *>(p.y) + tl.y_off + static_cast<int64_t>(32 * q) * p.n + c0;
        auto add_chunk = [&](const uint32_t(&v)[32], int c) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint8_t *row = stage_blk + lane * 64;
            const int xs = (lane >> 1) & 3;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4 *>(row + 16 * (j ^ xs)) =
                  make_uint4(v[16 * hf + 4 * j], v[16 * hf + 4 * j + 1], v[16 * hf + 4 * j + 2], v[16 * hf + 4 * j + 3]);
            __syncwarp();
            const int j = lane & 3;
            float4 o[4], add[4];
            float4 *dst[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = 8 * i + (lane >> 2);
              add[i] = *reinterpret_cast<const float4 *>(stage_blk + rr * 64 + 16 * (j ^ ((rr >> 1) & 3)));
              dst[i] = reinterpret_cast<float4 *>(ywarp + static_cast<int64_t>(rr) * p.n + 32 * c + 16 * hf + 4 * j);
              o[i] = *dst[i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[i].x = __fadd_rn(o[i].x, add[i].x);
              o[i].y = __fadd_rn(o[i].y, add[i].y);
              o[i].z = __fadd_rn(o[i].z, add[i].z);
              o[i].w = __fadd_rn(o[i].w, add[i].w);
              *dst[i] = o[i];
            }
            __syncwarp();
          }
        };
        add_chunk(v0, 0);
        add_chunk(v1, 1);
        add_chunk(v2, 2);
        add_chunk(v3, 3);
        continue;
      }
      const int warp_rows = tl.rows_valid - 32 * q;  // rows of this warp's 32 that are the expert's
      if (warp_rows > 0) {
        __nv_bfloat16 *ywarp = y + tl.y_off + static_cast<int64_t>(32 * q) * p.n + c0;
        auto emit = [&](const uint32_t(&v)[32], int c) {
          uint32_t packed[16];
          convert_chunk<K>(packed, v, sa, sw + 32 * c);
          store_block(ywarp + 32 * c, p.n, warp_rows, stage_blk, lane, packed);
        };
        emit(v0, 0);
        emit(v1, 1);
        emit(v2, 2);
        emit(v3, 3);
      }
    }
  }

  // Teardown: the pair meets once the leader's MMAs are drained and every
  // epilogue has read its accumulator; then both CTAs free tensor memory together.
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  pair::cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    pair::tmem_dealloc(tmem, kTmemCols);
  }
}

// Shared memory per CTA for the dynamic part (the static part is small).
constexpr int64_t kGemmSmemLimit = 227 * 1024 - 1024;

template <GemmKind K>
static cudaError_t launch_kind(const LaunchGemm &in) {
  using C = Cfg<K>;
  LaunchGemm a = in;
  a.stages = C::kStages;
  while (a.stages > 2 && gemm_smem_bytes(a.stages, C::kStageBytes, a.num_experts) > kGemmSmemLimit) --a.stages;
  const int smem_bytes = static_cast<int>(gemm_smem_bytes(a.stages, C::kStageBytes, a.num_experts));
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes);
  if (err != cudaSuccess) return err;
  int64_t bound;
  if (K == GemmKind::kWgradMxfp8)
    bound = static_cast<int64_t>(a.num_experts) * (a.m / kPairM) * (a.n / kBN);
  else
    bound = (a.m / kPairM + a.num_experts) * (a.n / kBN);
  int pairs = a.num_sms / 2;
  if (bound < pairs) pairs = static_cast<int>(bound > 0 ? bound : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<K>, a);
}

cudaError_t launch_grouped_gemm(const LaunchGemm &a) {
  switch (a.kind) {
    case GemmKind::kFwdNvfp4:
      return launch_kind<GemmKind::kFwdNvfp4>(a);
    case GemmKind::kDgradMxfp8:
      return launch_kind<GemmKind::kDgradMxfp8>(a);
    case GemmKind::kWgradMxfp8:
      return launch_kind<GemmKind::kWgradMxfp8>(a);
    case GemmKind::kFwdMxfp8:
      return launch_kind<GemmKind::kFwdMxfp8>(a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fme

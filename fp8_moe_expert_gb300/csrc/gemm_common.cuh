// gemm_common.cuh -- what the two grouped-GEMM kernels share: the 256 x 256 pair
// tile and its schedule over the experts, the group tables in shared memory, and
// the epilogue (accumulator out of tensor memory, per-token and per-column scales,
// bf16 out; or an fp32 accumulate for wgrad).
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1: the MoE
// layer's grouped GEMMs run as block-scaled tensor-core MMAs on Blackwell, NVFP4
// with a per-token FP32 scale applied in the GEMM epilogue for the forward, MXFP8
// for the backward.  "Scaling and Optimizing Frontier Model Training", "MXFP8
// expert kernels": grouped GEMMs over the experts' routed tokens.
//
// A pair of CTAs (a cluster of 2 on two SMs) computes 256 x 256 output tiles with
// cta_group::2 MMAs (M = 256: 128 rows in each CTA's tensor memory).  Each CTA
// stages its own 128 rows of A and its half (128 rows) of the tile's 256 B rows.
// Both CTAs walk the same tile sequence, derived in shared memory from the
// per-expert offsets: forward and dgrad go expert by expert, 256-row blocks of
// each expert's rows, 256-column blocks fastest; wgrad goes expert by expert in
// decreasing order of work (largest contraction first) and writes zeros for
// experts without rows.  Tiles are dealt out round-robin over the pairs, so the
// pairs that share a row block's A (or a column block's B) read it at about the
// same time (dealing a pair whole row blocks measured 4-6% slower).  There is no
// split over K: each output element is one accumulation, so a row's result does
// not depend on other rows.
#pragma once

#include "fme_device.cuh"
#include "fme_launch.h"

namespace fme {

constexpr int kBM = 128;           // rows per CTA
constexpr int kPairM = 256;        // rows per pair tile
constexpr int kBN = 256;           // columns per tile
constexpr int kHalfN = kBN / 2;    // B rows staged by each CTA
constexpr int kStageKBytes = 128;  // bytes of K per row per stage (one swizzle row)
constexpr int kMaxStages = 6;
constexpr int kOutBoxBytes = 32 * 32 * 2;                 // one 32-row x 32-column bf16 block
constexpr int kSwBytes = 128 * 4;                         // a warp's 128 column scales (forward)
constexpr int kOutBytes = 8 * (kOutBoxBytes + kSwBytes);  // staging block + column scales per epilogue warp
constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = kBM * kStageKBytes;
constexpr int kBBytes = kHalfN * kStageKBytes;
constexpr int kAccEmptyArrivals = 2 * 8;  // one per epilogue warp of the pair
// Shared memory per CTA for the dynamic part (the static part is small).
constexpr int64_t kGemmSmemLimit = 227 * 1024 - 1024;

// Elements of K per pipeline stage: one 128-byte swizzle row of codes.
__host__ __device__ constexpr int k_per_stage(GemmKind k) { return is_fwd_nvfp4(k) ? 256 : 128; }

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
  int32_t sfb_row;         // first of the two 128-row scale blocks of the tile's B rows
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
    tl.num_k = static_cast<int32_t>(p.k / k_per_stage(K));
    tl.rows_valid = static_cast<int32_t>(left < kBM ? left : kBM);
    tl.n0 = static_cast<int32_t>(nb * kBN);
    tl.y_off = r0 * p.n + nb * kBN;
    tl.a_y = static_cast<int32_t>(r0);
    tl.a_x0 = 0;
    tl.sfa_row = s.tiles[e] + static_cast<int32_t>(mb);
    tl.sfa_x0 = 0;
    if (K == GemmKind::kFwdNvfp4Swiglu) {
      // W_gu stacked as [gate rows (n / 2) | up rows (n / 2)] per expert: the leader
      // stages tile nb's 128 gate rows, the peer the matching 128 up rows, so that
      // accumulator columns 0-127 are gate and 128-255 up of the same 128 h columns;
      // their scale blocks (n / 256 blocks apart) are fetched one by one
      const int64_t brow = static_cast<int64_t>(e) * p.n + nb * kHalfN;
      tl.b_y = static_cast<int32_t>(brow + rank * (p.n / 2));
      tl.b_x0 = 0;
      tl.sfb_row = static_cast<int32_t>(brow / 128);
      tl.sfb_x0 = 0;
      tl.n0 = static_cast<int32_t>(nb * kHalfN);  // first h column
      tl.y_off = r0 * (p.n / 2) + nb * kHalfN;
    } else if (K == GemmKind::kFwdNvfp4 || K == GemmKind::kFwdMxfp8) {
      // B = stacked weights, expert e's rows e*n .. e*n+n-1, K contiguous; their
      // scales in the quantizers' tiled layout (one group: 128-row blocks in order)
      const int64_t brow = static_cast<int64_t>(e) * p.n + nb * kBN;
      tl.b_y = static_cast<int32_t>(brow + rank * kHalfN);
      tl.b_x0 = 0;
      tl.sfb_row = static_cast<int32_t>(brow / 128);
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

// Wait, on the leader, until every copy either CTA of the pair issued into one
// ring of stage barriers (`bars`, S stages) has landed.  The leader arms fill f
// of the ring (stage f % S, phase (f / S) & 1) for both CTAs' bytes; each CTA's
// copies complete on the leader's barrier.  `own` and `peer` are the fills each
// producer issued.  A fill is read by the MMAs only once both halves landed, and
// a producer reuses a stage only after the MMAs released it, so both counts lie
// in [c, c + S] for the c fills consumed, and only the latest fill of a stage can
// still be in flight.  After an abort the two counts may differ: a fill issued by
// the peer alone was never armed, so the leader arms it for the peer's bytes; a
// fill issued by the leader alone waits for peer bytes that will never come, so
// the leader counts them as arrived.  Each wait is bounded (kDrainLimitNs).
__device__ inline void drain_pair_ring(uint64_t *bars, int S, uint32_t own, uint32_t peer, uint32_t peer_bytes) {
  const uint32_t last = own > peer ? own : peer;
  for (uint32_t j = 0; j < static_cast<uint32_t>(S) && j < last; ++j) {
    const uint32_t f = j + S * ((last - 1 - j) / S);  // latest fill of stage j
    if (f >= own)
      mbar_arrive_expect_tx(&bars[j], peer_bytes);
    else if (f >= peer)
      mbar_complete_tx(&bars[j], peer_bytes);
    mbar_drain(&bars[j], (f / S) & 1);
  }
}

// The producers' hand-over at the end of their loops: the peer's producer sends
// its fill count to the leader (`fills_word` and `fills_bar` are the leader's
// shared word and barrier, initialised with one arrival); the leader's producer
// returns the peer's count, or its own if the count does not come within the
// time any of the peer's waits can take (reported as a time-out).
__device__ inline uint32_t exchange_fills(int rank, uint32_t filled, uint32_t *fills_word, uint64_t *fills_bar,
                                          int32_t *status) {
  if (rank != 0) {
    pair::st_remote_u32(pair::map_to_rank(fills_word, 0), filled);
    pair::arrive_remote_release(pair::map_to_rank(fills_bar, 0));
    return filled;
  }
  if (!pair::wait_acquire_cluster(fills_bar, 0, kWaitLimitNs + kDrainLimitNs)) {
    report(status, kDevTimeout);
    return filled;
  }
  return *reinterpret_cast<volatile uint32_t *>(fills_word);
}

// Build the tile tables (the same in both CTAs of a pair); returns false in
// every thread for malformed offsets.  `ok_flag` is a shared int.
template <GemmKind K>
__device__ bool prepare(const LaunchGemm &p, int *ok_flag, const Groups &g) {
  if (K != GemmKind::kWgradMxfp8) {
    if (!load_groups(g.off, g.tiles, p.offsets, p.num_experts, p.m, ok_flag)) return false;
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
    *ok_flag = ok ? 1 : 0;
  }
  __syncthreads();
  if (!*ok_flag) return false;
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

// SwiGLU of 32 consecutive h columns of one row: the gate and up accumulators
// scaled as the plain forward scales its outputs ((acc * S_x[t]) * S_w[n], fp32),
// h = silu(g) * u in fp32 (silu_times), rounded to bf16, two per word.  `swg` and
// `swu` point at the 32 gate and the 32 matching up column scales.
__device__ __forceinline__ void swiglu_chunk(uint32_t (&packed)[16], const uint32_t (&vg)[32],
                                             const uint32_t (&vu)[32], float sa, const float *swg, const float *swu) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 bg = *reinterpret_cast<const float2 *>(swg + 2 * j);
    const float2 bu = *reinterpret_cast<const float2 *>(swu + 2 * j);
    const float2 g = __fmul2_rn(
        __fmul2_rn(make_float2(__uint_as_float(vg[2 * j]), __uint_as_float(vg[2 * j + 1])), make_float2(sa, sa)), bg);
    const float2 u = __fmul2_rn(
        __fmul2_rn(make_float2(__uint_as_float(vu[2 * j]), __uint_as_float(vu[2 * j + 1])), make_float2(sa, sa)), bu);
    const __nv_bfloat162 h = __floats2bfloat162_rn(silu_times(g.x, u.x), silu_times(g.y, u.y));
    packed[j] = *reinterpret_cast<const uint32_t *>(&h);
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

// The same 32 x 32 block written by one bulk tensor store (every bf16 output; all
// rows of the block in the expert): the staging layout above is the 64-byte
// swizzle of the output map's 32 x 32 box (16-byte chunk j of row r at chunk
// j ^ ((r >> 1) & 3)).  Lane 0 issues the store; the block is rewritten only after
// the previous store has read it.  Measured against store_block: the MMA stages of
// the tile after an epilogue run up to 45% slower while the warps' global stores
// drain; with bulk stores gate/up tiles run 4% and down tiles 9% faster.
__device__ __forceinline__ void store_block_tma(const CUtensorMap *map, int32_t x, int32_t y, uint8_t *stage,
                                                int lane, const uint32_t (&packed)[16]) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  uint8_t *row = stage + lane * 64;
  const int s = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4 *>(row + 16 * (j ^ s)) =
        make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, x, y, stage);
    bulk_commit();
  }
}

// The epilogue of one warp (ew = 0..7 of the CTA's 8 epilogue warps, reading
// tensor-memory lane quarter q and column half ew / 4) over the pair's tiles.
// All 128 accumulator columns of a thread are loaded before the accumulator is
// released to the leader (a relaxed remote arrive: the data is in registers; a
// cluster-scope release made each arrive wait for the warp's earlier global
// stores, ~0.5 us per tile), then scaled, rounded and stored while the next
// tile's MMAs run.  acc_full / leader_acc_empty: the pair's accumulator barriers.
template <GemmKind K>
__device__ __forceinline__ void epilogue_warp(const LaunchGemm &p, const Groups &grp, int64_t pair_id, int64_t pairs,
                                              int64_t total, int rank, int ew, int q, int lane, uint32_t tmem,
                                              uint8_t *smem_out, uint64_t *acc_full, uint32_t leader_acc_empty,
                                              volatile int *abort_flag) {
  const int half = ew >> 2;
  const int r = q * 32 + lane;
  const int c0 = half * (kBN / 2);
  uint8_t *stage_blk = smem_out + ew * kOutBoxBytes;
  float *sw = reinterpret_cast<float *>(smem_out + 8 * kOutBoxBytes + ew * kSwBytes);
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
    if (is_fwd_nvfp4(K)) {
      if (valid) sa = __ldg(p.a_scale + tl.a_y + r);
      if (K == GemmKind::kFwdNvfp4Swiglu) {
        // lanes 0-15: the scales of this warp's 64 gate columns, lanes 16-31: of the matching up columns
        swv = __ldg(reinterpret_cast<const float4 *>(p.b_scale + static_cast<int64_t>(tl.e) * p.n + tl.n0 + half * 64 +
                                                     (lane >= 16 ? p.n / 2 : 0)) +
                    (lane & 15));
      } else {
        swv = __ldg(reinterpret_cast<const float4 *>(p.b_scale + static_cast<int64_t>(tl.e) * p.n + tl.n0 + c0) +
                    lane);
      }
    }
    if (!mbar_wait(acc_full, acc_phase, abort_flag, p.status)) break;
    tc_fence_after();
    uint32_t v0[32], v1[32], v2[32], v3[32];
    // v0, v1 from columns ta.., v2, v3 from tb..: this warp's 128 columns, or (SwiGLU)
    // its 64 gate columns and the matching 64 up columns
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t ta = K == GemmKind::kFwdNvfp4Swiglu ? tq + half * 64 : tq + c0;
    const uint32_t tb = K == GemmKind::kFwdNvfp4Swiglu ? tq + kHalfN + half * 64 : tq + c0 + 64;
    tmem_ld_32x32(ta, v0);
    tmem_ld_32x32(ta + 32, v1);
    tmem_ld_32x32(tb, v2);
    tmem_ld_32x32(tb + 32, v3);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) pair::arrive_remote_relaxed(leader_acc_empty);  // registers hold the data
    acc_phase ^= 1;
    if (is_fwd_nvfp4(K)) {
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
    // this CTA's first output row in map_y (wgrad: expert e's dW rows start at e * m)
    const int32_t out_row = K == GemmKind::kWgradMxfp8 ? static_cast<int32_t>(tl.e * p.m) + tl.a_y : tl.a_y;
    if (warp_rows > 0 && K == GemmKind::kFwdNvfp4Swiglu) {
      // h [rows x n / 2]: this warp's 64 h columns of the tile's 128
      const int64_t ldh = p.n / 2;
      const int oc0 = half * 64;
      __nv_bfloat16 *hwarp = y + tl.y_off + static_cast<int64_t>(32 * q) * ldh + oc0;
      auto emit_h = [&](const uint32_t(&vg)[32], const uint32_t(&vu)[32], int c) {
        uint32_t packed[16];
        swiglu_chunk(packed, vg, vu, sa, sw + 32 * c, sw + 64 + 32 * c);
        if (warp_rows >= 32) {
          store_block_tma(&p.map_y, tl.n0 + oc0 + 32 * c, out_row + 32 * q, stage_blk, lane, packed);
        } else {
          if (lane == 0) bulk_wait_read_all();  // a bulk store may still be reading the block
          __syncwarp();
          store_block(hwarp + 32 * c, ldh, warp_rows, stage_blk, lane, packed);
        }
      };
      emit_h(v0, v2, 0);
      emit_h(v1, v3, 1);
    } else if (warp_rows > 0) {
      __nv_bfloat16 *ywarp = y + tl.y_off + static_cast<int64_t>(32 * q) * p.n + c0;
      auto emit = [&](const uint32_t(&v)[32], int c) {
        uint32_t packed[16];
        convert_chunk<K>(packed, v, sa, sw + 32 * c);
        if (warp_rows >= 32) {
          store_block_tma(&p.map_y, tl.n0 + c0 + 32 * c, out_row + 32 * q, stage_blk, lane, packed);
        } else {
          if (lane == 0) bulk_wait_read_all();  // a bulk store may still be reading the block
          __syncwarp();
          store_block(ywarp + 32 * c, p.n, warp_rows, stage_blk, lane, packed);
        }
      };
      emit(v0, 0);
      emit(v1, 1);
      emit(v2, 2);
      emit(v3, 3);
    }
  }
  if (lane == 0) bulk_wait_all();  // the bulk stores are done before the CTA exits
}

// A pair-cluster launch of `kernel` on as many pairs as the work and the SMs allow.
template <typename Kernel>
cudaError_t launch_pairs(Kernel kernel, const LaunchGemm &a, int threads, int smem_bytes, int64_t tile_bound) {
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (err != cudaSuccess) return err;
  int pairs = a.num_sms / 2;
  if (tile_bound < pairs) pairs = static_cast<int>(tile_bound > 0 ? tile_bound : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Upper bound on the tiles of a call (work for at most that many pairs).
inline int64_t gemm_tile_bound(const LaunchGemm &a) {
  if (a.kind == GemmKind::kWgradMxfp8) return static_cast<int64_t>(a.num_experts) * (a.m / kPairM) * (a.n / kBN);
  return (a.m / kPairM + a.num_experts) * (a.n / kBN);
}

// The NVFP4 forward (gemm_nvfp4.cu).
cudaError_t launch_grouped_gemm_nvfp4(const LaunchGemm &a);

}  // namespace fme

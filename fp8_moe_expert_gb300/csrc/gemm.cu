// gemm.cu -- the MXFP8 grouped GEMMs (dgrad, wgrad and the MXFP8 forward) on the
// tcgen05 tensor cores, CTA pairs; and the dispatch of every grouped GEMM.
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1: MXFP8
// (E4M3 values, an E8M0 scale per 32) for the MoE backward, block-scaled MMAs on
// the tensor cores.  "Scaling and Optimizing Frontier Model Training", "MXFP8
// expert kernels": MXFP8 grouped GEMMs for the expert layers' forward and
// backward.
//
// One persistent kernel per call; the tile and its schedule are in
// gemm_common.cuh.  The scales reach tensor memory by tcgen05.cp from shared
// memory: one 128-K stage needs three 512-byte tile copies (A, B rows 0-127, B
// rows 128-255) for four MMAs, issued by two copier threads.  (Feeding them from
// registers with tcgen05.st, as the NVFP4 kernel does, measured 6-10% slower for
// these kinds: with one scale per 32 values the copies are few, and the extra
// warps cost more than they save.)  12 warps per CTA:
//   warp 0      TMA producer (both CTAs): A, B and their scale tiles into a
//               6-stage ring; every copy of the pair completes on a barrier of
//               the leader CTA, the scale tiles (issued first) on "sf_landed",
//               A and B on "full", so that the scale copies below overlap the
//               operand loads instead of following them;
//   warp 1      allocates 512 tensor-memory columns in both CTAs together; in the
//               leader, one thread issues the block-scaled MMAs
//               (kind::mxf8f6f4.block_scale.scale_vec::1X, M = 256, N = 256, the
//               scale id selecting the byte); one commit per two stages frees both
//               stages (and their scale buffers) in both CTAs, and at the end of a
//               tile a commit fills both CTAs' accumulators;
//   warps 10-11 in the leader, one thread of each copies its share of the
//               stage's three scale tiles into the stage's own tensor-memory
//               buffer (tcgen05.cp.cta_group::2.32x128b.warpx4: the copy
//               replicates a tile's 32 rows into all four lane quarters, which B
//               needs) ahead of the MMAs; a stage's tiles land only after both
//               producers saw the buffer's previous readers finish.
// Against a commit per stage and a separate scale-buffer ring: dgrad 2.40 ->
// 2.34 ms, wgrad 2.45 -> 2.38 ms on the 262144-row step.
//   warps 2-9   epilogue (both CTAs): see epilogue_warp.
#include "gemm_common.cuh"

namespace fme {

constexpr int kThreads = 384;    // producer, MMA, 8 epilogue warps, 2 scale copiers
constexpr int kCopierWarp = 10;  // and 11
constexpr int kCopiers = 2;
constexpr int kGroupBars = 4;   // ring of "group done" barriers (one commit per two stages)

struct CfgMx {
  static constexpr int kSfaBytes = 512;      // this CTA's 128 rows: one tile per 128-K stage
  static constexpr int kSfbBytes = 2 * 512;  // the tile's 256 B rows: two tiles
  static constexpr int kSfaCols = 4;         // tensor-memory columns per stage
  static constexpr int kSfbCols = 8;
  static constexpr int kSfCols = kSfaCols + kSfbCols;
  static constexpr int kStages = 6;  // ring depth when the shared memory allows
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  // Both CTAs' copies land on the leader's barriers: the operands on "full", the
  // scale tiles (issued first) on "sf_landed".
  static constexpr int kOperandTx = 2 * (kABytes + kBBytes);
  static constexpr int kScaleTx = 2 * (kSfaBytes + kSfbBytes);
  static_assert(kStages <= kMaxStages, "stage count");
  static_assert(kBN + kStages * kSfCols <= static_cast<int>(kTmemCols), "tensor memory budget");
};

struct SharedStateMx {
  uint64_t full[kMaxStages];       // the stage's A and B tiles have landed
  uint64_t sf_landed[kMaxStages];  // the stage's scale tiles have landed
  uint64_t sf_full[kMaxStages];   // the stage's scales are in its tensor-memory buffer (one arrival per copier)
  uint64_t grp_done[kGroupBars];  // the MMAs of fills 2c and 2c + 1 are done (both CTAs, by commit c)
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint64_t drain_cp[kCopiers];
  uint64_t peer_fills_bar;  // the peer's producer has written peer_fills (leader)
  uint32_t peer_fills;      // fills the peer's producer issued (leader)
  uint32_t tmem_base;
  int abort_flag;
  int ok_flag;
};

template <GemmKind K>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_mx_kernel(const __grid_constant__ LaunchGemm p) {
  using C = CfgMx;
  __shared__ SharedStateMx s;
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
  if (!prepare<K>(p, &s.ok_flag, grp)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.status, kDevBadOffsets);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.sf_landed[i], 1);
      mbar_init(&s.sf_full[i], kCopiers);
    }
    for (int i = 0; i < kGroupBars; ++i) mbar_init(&s.grp_done[i], 1);
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, kAccEmptyArrivals);
    mbar_init(&s.drain, 1);
    mbar_init(&s.peer_fills_bar, 1);
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
    uint32_t stage = 0;
    uint32_t filled = 0;  // stages filled so far (for the drain below)
    for (int64_t t = pair_id; t < total; t += pairs) {
      const Tile tl = tile_at<K>(p, grp, t, rank);
      // wgrad: the pairs' i-th tiles (a "wave") stream K forward for even i and
      // backward for odd i, so that a wave starts on the B panels' K range the
      // previous wave read last, which is still in L2 (a wave reads every B panel
      // of a large expert again).
      const bool reverse = K == GemmKind::kWgradMxfp8 && ((t / pairs) & 1);
      bool stop = false;
      for (int ks_ = 0; ks_ < tl.num_k; ++ks_) {
        const int ks = reverse ? tl.num_k - 1 - ks_ : ks_;
        // Fill f reuses the stage (and its tensor-memory scale buffer) of fill
        // f - S, whose MMAs commit (f - S) / 2 covers.
        if (filled >= static_cast<uint32_t>(S)) {
          const uint32_t c = (filled - S) >> 1;
          if (!mbar_wait<true>(&s.grp_done[c % kGroupBars], (c / kGroupBars) & 1, abort_flag, p.status)) {
            stop = true;
            break;
          }
        }
        // Scales first, on their own barrier: the copiers start on them while the
        // operands are still arriving, so the tensor-memory copies are done by the
        // time the MMAs could start.
        if (rank == 0) mbar_arrive_expect_tx(&s.sf_landed[stage], C::kScaleTx);
        const uint32_t sbar = pair::map_to_rank(&s.sf_landed[stage], 0);
        pair::tma_load_2d(smem_sfa + stage * C::kSfaBytes, &p.map_sfa, sbar, (tl.sfa_x0 + ks) * 64, tl.sfa_row);
        pair::tma_load_2d(smem_sfb + stage * C::kSfbBytes, &p.map_sfb, sbar, (tl.sfb_x0 + ks) * 64, tl.sfb_row);
        if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], C::kOperandTx);
        const uint32_t bar = pair::map_to_rank(&s.full[stage], 0);
        pair::tma_load_2d(smem_a + stage * kABytes, &p.map_a, bar, tl.a_x0 + ks * kStageKBytes, tl.a_y);
        pair::tma_load_2d(smem_b + stage * kBBytes, &p.map_b, bar, tl.b_x0 + ks * kStageKBytes, tl.b_y);
        ++filled;
        if (++stage == S) stage = 0;
      }
      if (stop) break;
    }
    // Every copy the pair issued lands before a CTA can exit (after an abort,
    // stages may be filled that no MMA will read).  All of them complete on the
    // leader's barriers: its producer drains both rings from both producers'
    // fill counts, before the teardown's cluster barrier releases the peer.
    const uint32_t peer = exchange_fills(rank, filled, &s.peer_fills, &s.peer_fills_bar, p.status);
    if (rank == 0) {
      drain_pair_ring(s.sf_landed, S, filled, peer, C::kSfaBytes + C::kSfbBytes);
      drain_pair_ring(s.full, S, filled, peer, kABytes + kBBytes);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------ MMA issuer (leader)
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    uint32_t fill = 0;  // fills consumed so far
    bool stop = false;
    const uint32_t sf_base = tmem + kBN;
    for (int64_t t = pair_id; t < total && !stop; t += pairs) {
      const Tile tl = tile_at<K>(p, grp, t, 0);
      if (tl.num_k == 0) continue;
      if (!mbar_wait<true>(&s.acc_empty, acc_phase ^ 1, abort_flag, p.status)) break;
      tc_fence_after();
      for (int ks = 0; ks < tl.num_k; ++ks) {
        if (!mbar_wait<true>(&s.full[stage], phase, abort_flag, p.status) ||
            !mbar_wait<true>(&s.sf_full[stage], phase, abort_flag, p.status)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = sf_base + stage * C::kSfCols;
        const uint32_t sfb_t = sfa_t + C::kSfaCols;
        const uint32_t a_s = smem_u32(smem_a + stage * kABytes);
        const uint32_t b_s = smem_u32(smem_b + stage * kBBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = desc_sw128_kmajor(a_s + kk * 32);
          const uint64_t bd = desc_sw128_kmajor(b_s + kk * 32);
          const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
          pair::mma_mxf8(tmem, ad, bd, pair::idesc_mxf8(kBN, kk), sfa_t, sfb_t, acc);
        }
        // one commit per two fills (see gemm_nvfp4.cu: a waited commit per four
        // MMAs costs the tensor pipe time)
        if (fill & 1) pair::commit_both(&s.grp_done[(fill >> 1) % kGroupBars]);
        ++fill;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (stop) break;
      pair::commit_both(&s.acc_full);
      acc_phase ^= 1;
    }
    // every tensor-core operation of the pair has finished before memory is released
    pair::commit_local(&s.drain);
    mbar_drain(&s.drain, 0);
  } else if (warp >= kCopierWarp && warp < kCopierWarp + kCopiers && lane == 0 && rank == 0) {
    // --------------------------------------------------- scale copiers (leader)
    // Copy each stage's three scale tiles (both CTAs, tcgen05.cp.cta_group::2)
    // into the next free tensor-memory buffer while the MMA issuer works on
    // earlier stages, then arrive on the buffer's "full" barrier.  Copier 0
    // takes A and B's rows 128-255, copier 1 B's rows 0-127.
    const int who = warp - kCopierWarp;
    uint32_t stage = 0, phase = 0;
    bool stop = false;
    const uint32_t sf_base = tmem + kBN;
    for (int64_t t = pair_id; t < total && !stop; t += pairs) {
      const Tile tl = tile_at<K>(p, grp, t, 0);
      for (int ks = 0; ks < tl.num_k; ++ks) {
        // The stage's scale tiles have landed, so both producers have seen the
        // MMAs of the stage's previous fill (the last readers of its buffer) finish.
        if (!mbar_wait<true>(&s.sf_landed[stage], phase, abort_flag, p.status)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = sf_base + stage * C::kSfCols;
        const uint32_t sfb_t = sfa_t + C::kSfaCols;
        const uint32_t sfa_s = smem_u32(smem_sfa + stage * C::kSfaBytes);
        const uint32_t sfb_s = smem_u32(smem_sfb + stage * C::kSfbBytes);
        if (who == 0) {
          pair::copy_scales(sfa_t, desc_scale_tile(sfa_s));
          pair::copy_scales(sfb_t + 4, desc_scale_tile(sfb_s + 512));
        } else {
          pair::copy_scales(sfb_t, desc_scale_tile(sfb_s));
        }
        pair::commit_local(&s.sf_full[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    pair::commit_local(&s.drain_cp[who]);
    mbar_drain(&s.drain_cp[who], 0);
  } else if (warp >= 2 && warp < kCopierWarp) {
    // --------------------------------------------------------------- epilogue
    epilogue_warp<K>(p, grp, pair_id, pairs, total, rank, warp - 2, warp & 3, lane, tmem, smem_out, &s.acc_full,
                     pair::map_to_rank(&s.acc_empty, 0), abort_flag);
  }

  // Teardown: the pair meets once the leader's MMAs and copies are drained and
  // every epilogue has read its accumulator; then both CTAs free tensor memory
  // together.
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

template <GemmKind K>
static cudaError_t launch_mx(const LaunchGemm &in) {
  using C = CfgMx;
  LaunchGemm a = in;
  a.stages = C::kStages;
  while (a.stages > 2 && gemm_smem_bytes(a.stages, C::kStageBytes, a.num_experts) > kGemmSmemLimit) --a.stages;
  const int smem_bytes = static_cast<int>(gemm_smem_bytes(a.stages, C::kStageBytes, a.num_experts));
  return launch_pairs(grouped_gemm_mx_kernel<K>, a, kThreads, smem_bytes, gemm_tile_bound(a));
}

cudaError_t launch_grouped_gemm(const LaunchGemm &a) {
  switch (a.kind) {
    case GemmKind::kFwdNvfp4:
    case GemmKind::kFwdNvfp4Swiglu:
      return launch_grouped_gemm_nvfp4(a);
    case GemmKind::kDgradMxfp8:
      return launch_mx<GemmKind::kDgradMxfp8>(a);
    case GemmKind::kWgradMxfp8:
      return launch_mx<GemmKind::kWgradMxfp8>(a);
    case GemmKind::kFwdMxfp8:
      return launch_mx<GemmKind::kFwdMxfp8>(a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fme

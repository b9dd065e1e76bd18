// gemm_nvfp4.cu -- the NVFP4 grouped GEMM of the forward, Y_e = X_e W_e^T, on the
// tcgen05 tensor cores (kind::mxf4nvf4.block_scale.scale_vec::4X, M = 256 over a
// CTA pair, N = 256, K = 64 per MMA), the per-token and per-column FP32 scales
// applied in the epilogue.  A second form (kFwdNvfp4Swiglu) runs the gate/up
// projection with h = silu(gate) * up formed in the epilogue: the leader stages a
// tile's gate rows, its peer the matching up rows (gemm_common.cuh, tile_at).
//
// "Composer 2 Technical Report" (papercache.org summary), section 6.1: the NVFP4
// variant of the MoE forward (E2M1 values, an E4M3 scale per 16-element block,
// an FP32 scale per token applied in the GEMM epilogue) on block-scaled
// tensor-core MMAs.
//
// The tile, its schedule and the epilogue are in gemm_common.cuh.  The block
// scales reach tensor memory through registers, not through tcgen05.cp: each
// copy instruction occupies the tensor core for about a third of an MMA whatever
// its size (measured: 21-26 ns per copy against 65 ns per M = 256, N = 256,
// K = 64 MMA), and a 256-deep stage of four MMAs needs six to eight copies (B's
// scales must sit in all four tensor-memory lane quarters), while tcgen05.st from
// the SM's registers does not occupy the tensor core at all (measured: 24 KB of
// stores per stage next to back-to-back MMAs left the MMA rate unchanged).  B's
// scales can then stay in the quantizers' tiled layout.  16 warps per CTA in
// four warpgroups:
//   warps 0-3   scale writers (both CTAs), warp w owning tensor-memory lane
//               quarter w: per stage, read the stage's scale tiles from shared
//               memory (where TMA put them), tcgen05.st them into the stage's own
//               tensor-memory scale buffer in the layout the MMA reads, and
//               arrive on the leader's "scales full" barrier;
//   warp 4      TMA producer (both CTAs): A, B and their scale tiles into a
//               5-stage ring; A and B complete on the leader's "full" barrier
//               (the leader's MMAs read both CTAs' tiles), the scale tiles on
//               this CTA's own "scales landed" barrier;
//   warp 5      allocates 512 tensor-memory columns in both CTAs together; in the
//               leader, one thread issues the MMAs; one commit per two stages
//               frees both stages (and their scale buffers) in both CTAs, and at
//               the end of a tile a commit fills both CTAs' accumulators;
//   warps 8-15  epilogue (both CTAs): see epilogue_warp.
// Why one commit per two stages: in a microbenchmark of back-to-back MMAs (128
// cycles per M = 256, N = 256, K = 64 MMA at 1.96 GHz), a wait on a commit issued
// one four-MMA stage earlier cost the pipe 100-150 ns per stage, however deep the
// ring, while one waited commit per eight MMAs cost nothing; without loads or
// scales this ring then runs at the MMA rate (measured 263 ns per stage).  A
// stage's tensor-memory scale buffer is free when the producer may refill the
// stage, so the writers wait only for the scale tiles to land.
// Registers: launched at 128 per thread; the writers and the producer/MMA
// warpgroup give some back (setmaxnreg) so that the epilogue holds its whole
// accumulator share (128 values per thread).
#include "gemm_common.cuh"

namespace fme {

namespace {

constexpr int kThreads = 512;  // 4 scale writers, producer, MMA, 2 idle, 8 epilogue warps
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kEpilogueWarp = 8;  // first of 8
constexpr int kGroupBars = 4;     // ring of "group done" barriers (one commit per two fills)
// Register budgets per thread (launch: 65536 / 512 = 128): writers, producer/MMA
// warpgroup, the two epilogue warpgroups; 128 * (96 + 64 + 2 * 176) = 65536.
constexpr uint32_t kRegsWriter = 96;
constexpr uint32_t kRegsControl = 64;
constexpr uint32_t kRegsEpilogue = 176;
static_assert(kRegsWriter + kRegsControl + 2 * kRegsEpilogue == 512, "register split must use the launch budget");
constexpr int kSfFullArrivals = 2 * 4;  // one per scale-writer warp of the pair

constexpr int kAtoms = 4;                   // 512-byte scale tiles per 128 rows per 256-deep stage
constexpr int kSfaBytes = 512 * kAtoms;     // this CTA's 128 A rows
constexpr int kSfbBytes = 2 * 512 * kAtoms;  // the tile's 256 B rows: [rows 0-127][rows 128-255]
constexpr int kStages = 5;                  // ring depth when the shared memory allows
constexpr int kSfBufs = kStages;            // one tensor-memory scale buffer per stage
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
// Tensor-memory scale ring after the 256 accumulator columns: all buffers' B
// columns (4 steps x 8), then all buffers' A columns (4 steps x 4), so that every
// tcgen05.st starts at a multiple of its width.
constexpr int kSfbCols = 32;
constexpr int kSfaCols = 16;
constexpr uint32_t kSfbBase = kBN;
constexpr uint32_t kSfaBase = kBN + kSfBufs * kSfbCols;
// A and B of both CTAs land on the leader's "full"; each CTA's scale tiles on its own "sf_landed".
constexpr int kOperandTx = 2 * (kABytes + kBBytes);
constexpr int kScaleTx = kSfaBytes + kSfbBytes;
static_assert(kStages <= kMaxStages, "ring size");
static_assert(kSfaBase + kSfBufs * kSfaCols <= kTmemCols, "tensor memory budget");

struct SharedState {
  uint64_t full[kMaxStages];       // the stage's A and B tiles (both CTAs) have landed (leader)
  uint64_t sf_landed[kMaxStages];  // this CTA's scale tiles of the stage have landed
  uint64_t sf_full[kMaxStages];    // every writer of the pair has stored the stage's scales (leader)
  uint64_t grp_done[kGroupBars];   // the MMAs of fills 2c and 2c + 1 are done (both CTAs, by commit c)
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint64_t peer_fills_bar;  // the peer's producer has written peer_fills (leader)
  uint32_t peer_fills;      // operand fills the peer's producer issued (leader)
  uint32_t tmem_base;
  int abort_flag;
  int ok_flag;
};

// One stage's scales from shared memory into tensor-memory buffer `b`, by the
// writer warp of lane quarter q (its 32 lanes).  The shared tiles are the
// quantizers' 512-byte tiles: row i (16 bytes) of a tile holds the four scale
// words of rows i, i + 32, i + 64, i + 96 of its 128-row block.  What the MMA
// reads (measured with a probe kernel that decoded which byte each output used):
//   A row r:    lane r, column (A base) + r / 32;
//   B column n: lane 32 q' + n % 32 for accumulator rows in every quarter q',
//               column (B base) + n / 32.
// So lane i of quarter q needs word q of its A tile row i (stored four times, so
// that column base + q holds it whatever q is), and all 16 bytes of row i of
// both B tiles (the same in every quarter).
__device__ __forceinline__ void write_scales(uint32_t tmem, int q, int lane, uint32_t b, const uint8_t *sfa_s,
                                             const uint8_t *sfb_s) {
  const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
  uint32_t va[16], vb[32];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(sfa_s + kk * 512 + lane * 16 + q * 4);
    va[4 * kk] = va[4 * kk + 1] = va[4 * kk + 2] = va[4 * kk + 3] = w;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = *reinterpret_cast<const uint4 *>(sfb_s + h * (512 * kAtoms) + kk * 512 + lane * 16);
      vb[8 * kk + 4 * h] = u.x;
      vb[8 * kk + 4 * h + 1] = u.y;
      vb[8 * kk + 4 * h + 2] = u.z;
      vb[8 * kk + 4 * h + 3] = u.w;
    }
  }
  tmem_st_32x32_x32(tmem + lanes + kSfbBase + b * kSfbCols, vb);
  tmem_st_32x32_x16(tmem + lanes + kSfaBase + b * kSfaCols, va);
}

// kKind: kFwdNvfp4, or kFwdNvfp4Swiglu (SwiGLU epilogue, h = silu(gate) * up).
template <GemmKind kKind>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_nvfp4_kernel(const __grid_constant__ LaunchGemm p) {
  __shared__ SharedState s;
  extern __shared__ uint8_t dyn_smem[];
  const int S = p.stages;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t *smem_a = smem;
  uint8_t *smem_b = smem_a + S * kABytes;
  uint8_t *smem_sfa = smem_b + S * kBBytes;
  uint8_t *smem_sfb = smem_sfa + S * kSfaBytes;
  uint8_t *smem_out = smem + ring_bytes(S, kStageBytes);
  int32_t *gmem = reinterpret_cast<int32_t *>(smem_out + kOutBytes);
  const Groups grp{gmem, gmem + (p.num_experts + 1), gmem + 2 * (p.num_experts + 1)};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(pair::cta_rank());
  const int64_t pair_id = blockIdx.x >> 1;
  const int64_t pairs = gridDim.x >> 1;

  // Both CTAs of a pair see the same offsets, so both return here or neither does.
  if (!prepare<kKind>(p, &s.ok_flag, grp)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.status, kDevBadOffsets);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.sf_landed[i], 1);
      mbar_init(&s.sf_full[i], kSfFullArrivals);
    }
    for (int i = 0; i < kGroupBars; ++i) mbar_init(&s.grp_done[i], 1);
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, kAccEmptyArrivals);
    mbar_init(&s.drain, 1);
    mbar_init(&s.peer_fills_bar, 1);
    s.abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
    prefetch_tensormap(&p.map_a);
    prefetch_tensormap(&p.map_b);
    prefetch_tensormap(&p.map_sfa);
    prefetch_tensormap(&p.map_sfb);
  }
  if (warp == kMmaWarp) {
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
  const int64_t total = total_tiles<kKind>(p, grp);

  if (warp < 4) {
    // ------------------------------------------------------------ scale writers
    regs_dec<kRegsWriter>();
    const int q = warp;
    const uint32_t leader_sf_full = pair::map_to_rank(&s.sf_full[0], 0);
    uint32_t stage = 0, phase = 0;
    bool stop = false;
    for (int64_t t = pair_id; t < total && !stop; t += pairs) {
      const Tile tl = tile_at<kKind>(p, grp, t, rank);
      for (int ks = 0; ks < tl.num_k; ++ks) {
        // The stage's scale tiles have landed, so the producer has seen the MMAs
        // of the stage's previous fill (the last readers of its tensor-memory
        // scale buffer) finish.
        if (!mbar_wait<true>(&s.sf_landed[stage], phase, abort_flag, p.status)) {
          stop = true;
          break;
        }
        tc_fence_after();
        write_scales(tmem, q, lane, stage, smem_sfa + stage * kSfaBytes, smem_sfb + stage * kSfbBytes);
        // The stores are complete in tensor memory once tcgen05.wait::st returns, and
        // the leader reads this buffer only after the barrier phase completes, so the
        // peer's arrive needs no memory ordering of its own: a cluster-scope release
        // there cost about 0.7 us per arrive (measured: the whole ring ran at one
        // stage per us), a relaxed arrive nothing measurable.
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&s.sf_full[stage]);
          else
            pair::arrive_remote_relaxed(leader_sf_full + stage * 8);
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp < kEpilogueWarp) {
    regs_dec<kRegsControl>();
    if (warp == kProducerWarp && lane == 0) {
      // -------------------------------------------------------------- producer
      uint32_t stage = 0;
      uint32_t filled = 0;  // stages filled so far (for the drain below)
      for (int64_t t = pair_id; t < total; t += pairs) {
        const Tile tl = tile_at<kKind>(p, grp, t, rank);
        bool stop = false;
        for (int ks = 0; ks < tl.num_k; ++ks) {
          // Fill f reuses the stage of fill f - S, whose MMAs commit (f - S) / 2 covers.
          if (filled >= static_cast<uint32_t>(S)) {
            const uint32_t c = (filled - S) >> 1;
            if (!mbar_wait<true>(&s.grp_done[c % kGroupBars], (c / kGroupBars) & 1, abort_flag, p.status)) {
              stop = true;
              break;
            }
          }
          // scale tiles first, on this CTA's own barrier: the writers start on them
          // while the operands are still arriving
          mbar_arrive_expect_tx(&s.sf_landed[stage], kScaleTx);
          const uint32_t sbar = pair::map_to_rank(&s.sf_landed[stage], rank);
          pair::tma_load_2d(smem_sfa + stage * kSfaBytes, &p.map_sfa, sbar, (tl.sfa_x0 + ks * kAtoms) * 64,
                            tl.sfa_row);
          if (kKind == GemmKind::kFwdNvfp4Swiglu) {
            // the gate and the up block of B's scales, n / 256 blocks apart
            pair::tma_load_2d(smem_sfb + stage * kSfbBytes, &p.map_sfb, sbar, (tl.sfb_x0 + ks * kAtoms) * 64,
                              tl.sfb_row);
            pair::tma_load_2d(smem_sfb + stage * kSfbBytes + kSfbBytes / 2, &p.map_sfb, sbar,
                              (tl.sfb_x0 + ks * kAtoms) * 64, tl.sfb_row + static_cast<int32_t>(p.n / 256));
          } else {
            pair::tma_load_2d(smem_sfb + stage * kSfbBytes, &p.map_sfb, sbar, (tl.sfb_x0 + ks * kAtoms) * 64,
                              tl.sfb_row);
          }
          if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], kOperandTx);
          const uint32_t bar = pair::map_to_rank(&s.full[stage], 0);
          pair::tma_load_2d(smem_a + stage * kABytes, &p.map_a, bar, tl.a_x0 + ks * kStageKBytes, tl.a_y);
          pair::tma_load_2d(smem_b + stage * kBBytes, &p.map_b, bar, tl.b_x0 + ks * kStageKBytes, tl.b_y);
          ++filled;
          if (++stage == S) stage = 0;
        }
        if (stop) break;
      }
      // Every copy this CTA issued lands before the CTA can exit (after an abort,
      // stages may be filled that no MMA will read).  The scale tiles complete on
      // this CTA's own barriers: wait for the last fill of each stage (fill f used
      // stage f % S in phase (f / S) & 1).  The operands complete on the leader's
      // barriers: its producer drains them from both producers' fill counts,
      // before the teardown's cluster barrier releases the peer.
      for (uint32_t j = 0; j < static_cast<uint32_t>(S) && j < filled; ++j)
        mbar_drain(&s.sf_landed[j], ((filled - 1 - j) / S) & 1);
      const uint32_t peer = exchange_fills(rank, filled, &s.peer_fills, &s.peer_fills_bar, p.status);
      if (rank == 0) drain_pair_ring(s.full, S, filled, peer, kABytes + kBBytes);
    } else if (warp == kMmaWarp && lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer (leader)
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      uint32_t fill = 0;  // fills consumed so far
      bool stop = false;
      for (int64_t t = pair_id; t < total && !stop; t += pairs) {
        const Tile tl = tile_at<kKind>(p, grp, t, 0);
        if (!mbar_wait<true>(&s.acc_empty, acc_phase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        for (int ks = 0; ks < tl.num_k; ++ks) {
          if (!mbar_wait<true>(&s.full[stage], phase, abort_flag, p.status) ||
              !mbar_wait<true>(&s.sf_full[stage], phase, abort_flag, p.status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + kSfaBase + stage * kSfaCols;
          const uint32_t sfb_t = tmem + kSfbBase + stage * kSfbCols;
          const uint32_t a_s = smem_u32(smem_a + stage * kABytes);
          const uint32_t b_s = smem_u32(smem_b + stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = desc_sw128_kmajor(a_s + kk * 32);
            const uint64_t bd = desc_sw128_kmajor(b_s + kk * 32);
            const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
            pair::mma_nvf4(tmem, ad, bd, pair::idesc_nvf4(kBN), sfa_t + 4 * kk, sfb_t + 8 * kk, acc);
          }
          // One commit per two fills: waiting on a commit costs the tensor pipe time
          // unless the MMAs of about two stages separate it from the wait.
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
    }
  } else {
    // ----------------------------------------------------------------- epilogue
    regs_inc<kRegsEpilogue>();
    epilogue_warp<kKind>(p, grp, pair_id, pairs, total, rank, warp - kEpilogueWarp, warp & 3, lane, tmem, smem_out,
                         &s.acc_full, pair::map_to_rank(&s.acc_empty, 0), abort_flag);
  }

  // Teardown: the pair meets once the leader's MMAs are drained, every copy has
  // landed and every epilogue has read its accumulator; then both CTAs free
  // tensor memory together.  (Nothing but `tmem` is used past the roles: a value
  // live across them would hold a register in every role's loop.)
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  pair::cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    pair::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

template <GemmKind K>
cudaError_t launch_gemm_nvfp4_kind(const LaunchGemm &in) {
  LaunchGemm a = in;
  a.stages = kStages;
  while (a.stages > 2 && gemm_smem_bytes(a.stages, kStageBytes, a.num_experts) > kGemmSmemLimit) --a.stages;
  const int smem_bytes = static_cast<int>(gemm_smem_bytes(a.stages, kStageBytes, a.num_experts));
  // The warpgroups' register budgets add up to exactly 128 per thread: a kernel
  // built with fewer registers at launch would leave the epilogue's increase
  // waiting forever, so it is never launched.
  cudaFuncAttributes fa{};
  cudaError_t err = cudaFuncGetAttributes(&fa, grouped_gemm_nvfp4_kernel<K>);
  if (err != cudaSuccess) return err;
  if (fa.numRegs != 65536 / kThreads) return cudaErrorInvalidConfiguration;
  return launch_pairs(grouped_gemm_nvfp4_kernel<K>, a, kThreads, smem_bytes, gemm_tile_bound(a));
}

cudaError_t launch_grouped_gemm_nvfp4(const LaunchGemm &in) {
  return in.kind == GemmKind::kFwdNvfp4Swiglu ? launch_gemm_nvfp4_kind<GemmKind::kFwdNvfp4Swiglu>(in)
                                              : launch_gemm_nvfp4_kind<GemmKind::kFwdNvfp4>(in);
}

}  // namespace fme

// fme_device.cuh -- device-side building blocks shared by the kernels of libfme.so:
// inline PTX for mbarriers, TMA bulk copies and the tcgen05 tensor-core path
// (tensor memory allocation, scale-factor copies, block-scaled MMA, loads),
// bounded waits, the tiled scale-factor address, and group (expert) lookup.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fme {

// Bits OR-ed into the caller's device status word (mirror FME_DEV_* in fme.h).
constexpr int kDevTimeout = 0x1;
constexpr int kDevBadOffsets = 0x2;
constexpr int kDevBadIndex = 0x4;
constexpr int kMaxGroups = 1024;

// A bounded wait gives up after this long (ns of %globaltimer); real waits in
// these kernels last microseconds to a fraction of a millisecond.  A test build
// may shorten it (-DFME_WAIT_LIMIT_NS=...) so that waits run out on purpose; the
// waits that drain copies and MMAs already in flight before a CTA exits keep
// their own, fixed limit (kDrainLimitNs), so the shortened build still lets
// that work land.
#ifndef FME_WAIT_LIMIT_NS
#define FME_WAIT_LIMIT_NS 2000000000ull
#endif
#ifndef FME_WAIT_SPINS
#define FME_WAIT_SPINS 32
#endif
constexpr uint64_t kWaitLimitNs = FME_WAIT_LIMIT_NS;
constexpr int kWaitSpins = FME_WAIT_SPINS;  // barrier polls between two reads of the clock
constexpr uint64_t kDrainLimitNs = 2000000000ull;
// Longest a single barrier poll may suspend its thread (below the shortest wait
// limit a test build uses, so that limit is still honoured to within a poll).
constexpr uint32_t kPollSuspendNs = kWaitLimitNs < 1000000ull ? static_cast<uint32_t>(kWaitLimitNs) : 1000000u;

__device__ __forceinline__ void report(int32_t *status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ fp32 arithmetic --
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// silu(g) * u in fp32 (SwiGLU, h = silu(gate) * up), sigma in the form that cannot
// overflow: t = e^-|g| (the square of e^(-|g|/2), so that it rounds into the
// subnormal range instead of flushing while g e^g is still representable),
// sigma = (g >= 0 ? 1 : t) / (1 + t).  Relative error a few 2^-17 at most (the
// fast exponential), far below bf16's.
__device__ __forceinline__ float silu_times(float g, float u) {
  const float s = __expf(-0.5f * fabsf(g));
  const float t = s * s;
  const float sig = (g >= 0.0f ? 1.0f : t) * rcp_approx(1.0f + t);
  return g * sig * u;
}

// ------------------------------------------------------------------ mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Counts `bytes` of the current phase's transaction as arrived without any copy
// (for bytes that were expected but will never be sent).
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// The same poll with a suspend-time hint: the thread may sleep until the phase
// completes (the hardware wakes it then), for at most kPollSuspendNs.  Measured
// on the NVFP4 GEMM: 3-4% faster than polls without the hint.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kPollSuspendNs)
      : "memory");
  return done != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up when
// *abort is set by another thread or after kWaitLimitNs; on a time-out it sets
// *abort and reports kDevTimeout.  Returns true when the phase completed.
template <bool kSuspend = false>
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int32_t *status) {
  auto poll = [&] { return kSuspend ? mbar_try_wait_suspend(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < kWaitSpins; ++i)
      if (poll()) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1;
      report(status, kDevTimeout);
      return false;
    }
  }
}

// Wait for the phase of `bar` with the given parity, up to kDrainLimitNs, with no
// abort flag: used at the end of a role to let copies or MMAs already issued land.
__device__ __forceinline__ bool mbar_drain(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kDrainLimitNs) return false;
  return true;
}

// ----------------------------------------------------------------- TMA copies --
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tile store from this CTA's shared memory (bulk-group completion).  The
// coordinates must keep x * element size a multiple of 16 bytes and be >= 0.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int32_t x, int32_t y, const void *src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's committed bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The issuing thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (quarter base + i).
__device__ __forceinline__ void tmem_ld_32x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x N consecutive 32-bit columns from registers: thread i writes lane
// (quarter base + i).  The first column must be a multiple of N.
__device__ __forceinline__ void tmem_st_32x32_x4(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}

__device__ __forceinline__ void tmem_st_32x32_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st_32x32_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Per-warpgroup register budgets (every warp of a warpgroup executes the same one).
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Shared-memory matrix descriptor, K-major operand tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked
// along M/N (stride 1024), descriptor version 1 (bit 46), layout code 2 = 128B swizzle.
__device__ __forceinline__ uint64_t desc_sw128_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(16 >> 4) << 16;    // leading offset: unused for this layout
  d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride offset: next 8-row group
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Descriptor of a 512-byte scale tile for tcgen05.cp: no swizzle, 8-row x 16-byte
// core matrices packed every 128 bytes along the rows.
__device__ __forceinline__ uint64_t desc_scale_tile(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// ---------------------------------------------------------- scale-tile layout --
// Byte offset of scale (pr, c) in the tiled layout with C4 scales per padded row.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t pr, int64_t c, int64_t c4) {
  return ((pr >> 7) * (c4 >> 2) + (c >> 2)) * 512 + (pr & 31) * 16 + ((pr & 127) >> 5) * 4 + (c & 3);
}

// ------------------------------------------------------------ group lookup --
// Shared-memory copy of a group partition: off[g] row offsets and tiles[g] =
// sum_{g'<g} ceil(n_g'/128) (so padded row = 128 * tiles[g] + local row).
struct GroupTable {
  int32_t off[kMaxGroups + 1];
  int32_t tiles[kMaxGroups + 1];
};

// Load and check `offsets` (NULL = one group of `rows`) into off[0..G] and the
// running 128-row tile counts into tiles[0..G]; the whole block calls it.
// Returns false (same value in every thread) if the offsets do not rise from 0
// to rows.
__device__ inline bool load_groups(int32_t *off, int32_t *tiles, const int32_t *offsets, int32_t num_groups,
                                   int64_t rows, int *flag) {
  if (threadIdx.x == 0) {
    bool ok = true;
    int32_t acc = 0;
    int32_t prev = 0;
    for (int g = 0; g <= num_groups; ++g) {
      int32_t v = offsets ? __ldg(offsets + g) : (g == 0 ? 0 : static_cast<int32_t>(rows));
      if (g == 0 && v != 0) ok = false;
      if (g > 0) {
        if (v < prev) ok = false;
        int32_t n = v - prev;
        tiles[g - 1] = acc;
        acc += (n > 0 ? (n + 127) / 128 : 0);
      }
      off[g] = v;
      prev = v;
    }
    tiles[num_groups] = acc;
    if (prev != rows) ok = false;
    *flag = ok ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

__device__ inline bool load_groups(GroupTable &t, const int32_t *offsets, int32_t num_groups, int64_t rows,
                                   int *flag) {
  return load_groups(t.off, t.tiles, offsets, num_groups, rows, flag);
}

// Group holding row r: the last g with off[g] <= r (skipping empty groups).
__device__ __forceinline__ int find_group(const int32_t *off, int num_groups, int64_t r) {
  int lo = 0, hi = num_groups;  // off[lo] <= r < off[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (off[mid] <= r)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// ------------------------------------------------------ CTA pairs (clusters) --
namespace pair {

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

// All threads of both CTAs.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Relaxed: orders no memory operation.  Used only to hand tensor memory back
// after tcgen05.wait::ld, when nothing the waiter does depends on this thread's
// memory writes; a release at cluster scope would first wait for all of the
// thread's earlier global stores (measured: ~0.5 us per tile of the forward GEMM).
__device__ __forceinline__ void arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Store to a 32-bit word of another CTA's shared memory; the reader sees it after
// a barrier phase completed by arrive_remote_release and observed by
// wait_acquire_cluster.
__device__ __forceinline__ void st_remote_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Arrive on another CTA's barrier after this thread's earlier memory operations
// (release at cluster scope).
__device__ __forceinline__ void arrive_remote_release(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Wait, up to limit_ns, for the phase of this CTA's barrier `bar` with the given
// parity, acquiring at cluster scope what the arriving CTAs released.
__device__ __forceinline__ bool wait_acquire_cluster(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// 2-D tile load into this CTA's shared memory whose completion is counted on the
// mbarrier at `bar_cluster_addr` (the leader CTA's barrier).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint32_t bar_cluster_addr, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(x), "r"(y)
      : "memory");
}

// Tensor memory: allocated, released and freed by one warp of each CTA of the pair together.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Issued by the leader: each CTA's 512-byte scale tile (same shared address)
// into four tensor-memory columns of that CTA, replicated over the lane quarters.
__device__ __forceinline__ void copy_scales(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Arrive on the mbarrier at the same shared offset in both CTAs when the
// leader's tensor-core operations issued so far are done.
__device__ __forceinline__ void commit_both(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

__device__ __forceinline__ void commit_local(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// D (+)= A * B^T over the pair: M = 256 (128 rows in each CTA), E4M3 operands,
// one E8M0 scale per 32 K.
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Same with packed E2M1 operands and one E4M3 scale per 16 K.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptors for M = 256 (the pair), N = n.
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t n, uint32_t sf_id) {
  return (sf_id << 4) | (0u << 7) | (0u << 10) | ((n >> 3) << 17) | (1u << 23) | ((256u >> 4) << 24) |
         (sf_id << 29);
}

__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (0u << 23) | ((256u >> 4) << 24);
}

}  // namespace pair

}  // namespace fme

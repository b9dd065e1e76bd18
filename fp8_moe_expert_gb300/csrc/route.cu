// route.cu -- grouping routed tokens by expert, and combining the experts' rows.
//
// "Cursor Composer 2 report deep dive", section 2, and "Composer 2 Technical
// Report" (papercache.org summary), section 6.1: the routed tokens are quantized
// before they are dispatched to their experts, and the experts' outputs are
// combined per token in BF16.  Section 6.2 of the report: the expert choices are
// replayed from the inference engine ("router replay"), so the grouping must be a
// pure function of the per-token top-k expert ids.  The grouping here is a stable
// counting sort: assignment a = t * top_k + k of token t goes to expert ids[a],
// and the assignments of one expert keep their order of a.  Grouped row r therefore depends only on the ids,
// never on scheduling.
//
// Three launches over chunks of kRouteChunk assignments:
//   1. per-chunk histograms of the expert ids into the workspace [chunks x E];
//   2. one CTA turns them into per-(chunk, expert) start rows and the offsets;
//   3. every chunk places its assignments: within a warp, lanes with the same
//      expert are ranked with __match_any_sync; warps go in order, each adding its
//      counts to a per-expert running total in shared memory.
// Ids outside [0, E) are reported (FME_DEV_BAD_INDEX), get row_of = -1 and take
// no grouped row.
#include "fme_device.cuh"
#include "fme_launch.h"

namespace fme {

constexpr int kRouteChunk = 1024;  // assignments per chunk = threads per CTA

__global__ void __launch_bounds__(kRouteChunk) route_hist_kernel(const int32_t *__restrict__ ids, int64_t n,
                                                                 int num_experts, int32_t *__restrict__ ws,
                                                                 int32_t *status) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < num_experts; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t a = static_cast<int64_t>(blockIdx.x) * kRouteChunk + threadIdx.x;
  if (a < n) {
    const int32_t e = __ldg(ids + a);
    if (e >= 0 && e < num_experts)
      atomicAdd(&hist[e], 1);
    else
      report(status, kDevBadIndex);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < num_experts; e += blockDim.x)
    ws[static_cast<int64_t>(blockIdx.x) * num_experts + e] = hist[e];
}

// One CTA of 1024 threads turns the per-chunk counts into start rows.  Thread t <
// S * E (S = 1024 / E slices of the chunks) owns expert e = t % E over slice
// j = t / E, so every pass over the workspace reads rows of E consecutive words.
//   pass 1: each thread sums its slice -> part[j][e];
//   then thread e scans part[.][e] over the slices (exclusive) into its total,
//   the totals are scanned over the experts into the offsets, and part[j][e]
//   becomes the first grouped row of slice j's assignments to expert e;
//   pass 2: each thread walks its slice, replacing ws[c][e] by its start row.
__global__ void __launch_bounds__(1024) route_scan_kernel(int64_t chunks, int num_experts, int32_t *__restrict__ ws,
                                                          int32_t *__restrict__ offsets) {
  __shared__ int32_t part[1024];
  __shared__ int32_t warp_sum[32];
  const int t = threadIdx.x;
  const int E = num_experts;
  const int S = 1024 / E;
  const int64_t per = (chunks + S - 1) / S;
  const bool owner = t < S * E;
  const int e_t = owner ? t % E : 0;
  const int j_t = owner ? t / E : 0;
  const int64_t c_lo = min(chunks, static_cast<int64_t>(j_t) * per);
  const int64_t c_hi = min(chunks, c_lo + per);
  if (owner) {
    int32_t sum = 0;
    for (int64_t c = c_lo; c < c_hi; ++c) sum += ws[c * E + e_t];
    part[t] = sum;
  }
  __syncthreads();
  // thread e: exclusive scan over the slices, total of expert e
  int32_t total = 0;
  if (t < E) {
    for (int j = 0; j < S; ++j) {
      const int32_t v = part[j * E + t];
      part[j * E + t] = total;
      total += v;
    }
  }
  // exclusive scan of the totals over the experts
  const int lane = t & 31, warp = t >> 5;
  int32_t incl = total;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const int32_t up = __shfl_up_sync(0xFFFFFFFFu, incl, s);
    if (lane >= s) incl += up;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_sum[lane];
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int32_t up = __shfl_up_sync(0xFFFFFFFFu, w, s);
      if (lane >= s) w += up;
    }
    warp_sum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  if (t < E) {
    const int32_t excl = incl - total + (warp > 0 ? warp_sum[warp - 1] : 0);
    offsets[t] = excl;
    if (t == E - 1) offsets[E] = excl + total;
    for (int j = 0; j < S; ++j) part[j * E + t] += excl;
  }
  __syncthreads();
  if (owner) {
    int32_t run = part[t];
    for (int64_t c = c_lo; c < c_hi; ++c) {
      const int32_t v = ws[c * E + e_t];
      ws[c * E + e_t] = run;
      run += v;
    }
  }
}

__global__ void __launch_bounds__(kRouteChunk) route_scatter_kernel(const int32_t *__restrict__ ids, int64_t n,
                                                                    int num_experts,
                                                                    const int32_t *__restrict__ ws,
                                                                    int32_t *__restrict__ row_of,
                                                                    int32_t *__restrict__ src_row) {
  extern __shared__ int32_t run[];
  for (int e = threadIdx.x; e < num_experts; e += blockDim.x) run[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t a = static_cast<int64_t>(blockIdx.x) * kRouteChunk + threadIdx.x;
  int32_t e = -1;
  if (a < n) {
    e = __ldg(ids + a);
    if (e < 0 || e >= num_experts) e = -1;
  }
  const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(same & ((1u << lane) - 1u));
  const bool leader = rank == 0;
  const int32_t *base = ws + static_cast<int64_t>(blockIdx.x) * num_experts;
  for (int w = 0; w < (kRouteChunk >> 5); ++w) {
    if (warp == w && e >= 0) {
      const int32_t dest = base[e] + run[e] + rank;
      __syncwarp(same);
      if (leader) run[e] += __popc(same);
      row_of[a] = dest;
      src_row[dest] = static_cast<int32_t>(a);
    }
    __syncthreads();
  }
  if (a < n && e < 0) row_of[a] = -1;
}

// Per-(chunk, expert) counters for routing calls that bring no workspace: 4 MB
// of device memory that exists for the module's lifetime, so such a call makes
// no allocation.  Calls that use it must be ordered (one stream, or events).
__device__ int32_t g_route_counters[kRouteStaticWords];

cudaError_t launch_route_static(LaunchRoute r) {
  void *p = nullptr;
  cudaError_t err = cudaGetSymbolAddress(&p, g_route_counters);
  if (err != cudaSuccess) return err;
  r.ws = static_cast<int32_t *>(p);
  return launch_route(r);
}

cudaError_t launch_route(const LaunchRoute &r) {
  const int64_t n = r.tokens * r.top_k;
  const int64_t chunks = (n + kRouteChunk - 1) / kRouteChunk;
  const size_t hist_smem = static_cast<size_t>(r.num_experts) * sizeof(int32_t);
  if (chunks > 0) {
    route_hist_kernel<<<static_cast<unsigned>(chunks), kRouteChunk, hist_smem, r.stream>>>(r.ids, n, r.num_experts,
                                                                                          r.ws, r.status);
  }
  route_scan_kernel<<<1, 1024, 0, r.stream>>>(chunks, r.num_experts, r.ws, r.offsets);
  if (chunks > 0) {
    route_scatter_kernel<<<static_cast<unsigned>(chunks), kRouteChunk, hist_smem, r.stream>>>(
        r.ids, n, r.num_experts, r.ws, r.row_of, r.src_row);
  }
  return cudaGetLastError();
}

// out[t, :] = bf16(sum_k w[t, k] * y[row_of[t*top_k + k], :]) in fp32, k in order,
// each product and sum rounded separately; assignments with row_of < 0 are
// skipped.  One warp per token row, 8 columns per lane per step; the rows of
// kCombineBatch assignments are loaded before they are summed (in order), so a
// lane keeps that many 16-byte loads in flight.
constexpr int kCombineBatch = 4;

__global__ void __launch_bounds__(256) moe_combine_kernel(const uint16_t *__restrict__ y, const int32_t *__restrict__ row_of,
                                                          const float *__restrict__ weights, int64_t tokens,
                                                          int top_k, int n, int64_t rows_y, uint16_t *__restrict__ out,
                                                          int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < tokens;
       t += warps) {
    const int32_t *rt = row_of + t * top_k;
    const float *wt = weights + t * top_k;
    bool bad = false;
    for (int c0 = lane * 8; c0 < n; c0 += 256) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int k0 = 0; k0 < top_k; k0 += kCombineBatch) {
        uint4 v[kCombineBatch];
        float w[kCombineBatch];
        bool use[kCombineBatch];
#pragma unroll
        for (int b = 0; b < kCombineBatch; ++b) {
          const int k = k0 + b;
          const int32_t r = (k < top_k) ? __ldg(rt + k) : -1;
          use[b] = r >= 0 && r < rows_y;
          bad |= r >= rows_y;
          w[b] = use[b] ? __ldg(wt + k) : 0.0f;
          v[b] = use[b] ? __ldg(reinterpret_cast<const uint4 *>(y + static_cast<int64_t>(r) * n + c0))
                        : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int b = 0; b < kCombineBatch; ++b) {
          if (!use[b]) continue;
          const uint32_t wd[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w[b], __uint_as_float(wd[i] << 16)));
            acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w[b], __uint_as_float(wd[i] & 0xFFFF0000u)));
          }
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t *>(&b);
      }
      *reinterpret_cast<uint4 *>(out + t * n + c0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (bad) report(status, kDevBadIndex);
  }
}

cudaError_t launch_combine(const LaunchCombine &c) {
  const int64_t need = (c.tokens + 7) / 8;
  const int64_t cap = static_cast<int64_t>(c.num_sms) * 8;
  const int blocks = static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
  moe_combine_kernel<<<blocks, 256, 0, c.stream>>>(static_cast<const uint16_t *>(c.y), c.row_of, c.weights, c.tokens,
                                                   c.top_k, static_cast<int>(c.n), c.rows_y,
                                                   static_cast<uint16_t *>(c.out), c.status);
  return cudaGetLastError();
}

}  // namespace fme

/*
 * fme.h -- C ABI of the GB300 low-precision MoE expert path (libfme.so).
 *
 * Five calls, named after the operations of the MoE expert layer (plus a fused
 * row-wise + column-wise MXFP8 quantizer for tensors needed both ways):
 *   quantize_nvfp4_pertoken   NVFP4 variant of the forward: E2M1 codes, one E4M3
 *                             scale per 16 values along K, one FP32 scale per token.
 *   quantize_nvfp4_pertensor  standard NVFP4 (one FP32 scale per tensor), the comparator.
 *   swiglu_quantize_nvfp4     silu(gate) * up of the gate/up output, quantized as above.
 *   moe_route (moe_route_noalloc), permute_quantize_nvfp4, permute_quantize_mxfp8,
 *   moe_combine               grouping the routed tokens by expert (quantizing
 *                             them in grouped order) and combining the experts'
 *                             outputs per token.
 *   quantize_mxfp8            standard MXFP8 of the backward: E4M3 codes, one E8M0
 *                             scale per 32 values, row-wise or column-wise.
 *   swiglu_backward_quantize_mxfp8   the SwiGLU backward, d(gate/up) quantized
 *                             row-wise and column-wise for the gate/up gradients.
 *   grouped_gemm_fwd_nvfp4    Y_e = X_e W_e^T per expert, per-token scales applied
 *                             in the epilogue, bf16 out.
 *   grouped_gemm_fwd_nvfp4_swiglu   the gate/up projection of the same product with
 *                             h = silu(gate) * up formed in the epilogue, bf16 h out.
 *   grouped_gemm_fwd_mxfp8    the same product with MXFP8 operands (no per-token scale).
 *   grouped_gemm_dgrad_mxfp8  dX_e = dY_e W_e per expert, bf16 out.
 *   grouped_gemm_wgrad_mxfp8  dW_e = dY_e^T H_e per expert, bf16 out (or added into
 *                             fp32: grouped_gemm_wgrad_mxfp8_accumulate).
 *
 * Source passages ("Composer 2 Technical Report", papercache.org summary,
 * section 6.1): the NVFP4-variant paragraph (E2M1, E4M3 per block of 16, FP32
 * per token, scale applied at the cost of quantize and GEMM-epilogue latency),
 * the MXFP8-backward paragraph (E4M3 values, E8M0 scale per 32), the
 * hardware-math paragraph (IEEE-compliant division when quantizing NVFP4), and
 * the block-scaled tensor-core GEMM sentence (dequantization inside the
 * systolic-array multiply).  "Scaling and Optimizing Frontier Model Training",
 * "MXFP8 expert kernels": native block-scaled grouped GEMMs for expert shapes
 * (32 experts per rank, hidden 7168, intermediate 2048).
 *
 * Conventions for every call
 *   - Pointers are device pointers, allocated and owned by the caller.  The
 *     library allocates nothing, frees nothing and never synchronises a stream
 *     (except fme_read_device_status, which says so).
 *   - Every call enqueues its work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns at once.
 *   - Arguments are checked on the host before anything is launched; a failed
 *     check returns its status and launches nothing.
 *   - bf16 tensors are row-major with the last dimension contiguous.  Every
 *     pointer must be 16-byte aligned.
 *   - Inputs must be finite; NaN or Inf inputs are outside the contract.
 *   - Errors the kernels detect (malformed offsets, an index out of range, a
 *     bounded wait that ran out) are OR-ed as FME_DEV_* bits into `dev_status`, a
 *     caller-owned device int32 that the caller zeroes; dev_status may be NULL to
 *     ignore them.  A kernel that finds malformed offsets or runs out of time
 *     writes nothing more and returns; an out-of-range index is skipped (or read
 *     as row 0, where the call says so) and the rest of the work completes.
 *   - Calls are thread-safe and keep no per-call state, except moe_route_noalloc,
 *     whose counters are one static device array: its calls must be ordered.
 *
 * Grouped rows (experts)
 *   `offsets` is a device int32 array of num_groups + 1 non-decreasing prefix
 *   sums, offsets[0] = 0 and offsets[num_groups] = rows: group g owns rows
 *   [offsets[g], offsets[g+1]).  NULL means one group holding every row.
 *
 * Scale-factor layout (this library's contract; the pages give none)
 *   A scale matrix with logical shape [R x C] (R rows of the quantized tensor,
 *   C = cols / block) is stored padded: each group's rows start at a multiple
 *   of 128 (padded row pr = 128 * sum_{g'<g} ceil(n_g'/128) + local row), and
 *   C is rounded up to C4 = 4 * ceil(C / 4).  Element (pr, c) lives at byte
 *      ((pr / 128) * (C4 / 4) + c / 4) * 512 + (pr % 32) * 16 + ((pr % 128) / 32) * 4 + c % 4
 *   i.e. 512-byte tiles of 128 rows x 4 scales, the order in which the tensor
 *   core's block-scale operand is copied into tensor memory.  Bytes of padding
 *   rows are left unwritten; a row's padding columns (C <= c < C4, only when C is
 *   not a multiple of 4) are written as 0, with the row's last four scales.
 *   fme_sf_bytes() gives the buffer size.
 */
#ifndef FME_H
#define FME_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t fme_status;

#define FME_OK 0
#define FME_ERR_INVALID_ARGUMENT 1   /* null pointer, negative size, bad axis  */
#define FME_ERR_MISALIGNED 2         /* a pointer or a leading dimension not 16-byte aligned */
#define FME_ERR_UNSUPPORTED_SHAPE 3  /* a size outside the supported tiling (see each call) */
#define FME_ERR_UNSUPPORTED_DEVICE 4 /* the current device is not compute capability 10.3 */
#define FME_ERR_CUDA 5               /* a CUDA runtime or driver call failed; see fme_last_cuda_error() */
#define FME_ERR_DEVICE_TIMEOUT 6     /* reported by fme_read_device_status() */
#define FME_ERR_DEVICE_BAD_OFFSETS 7 /* reported by fme_read_device_status() */
#define FME_ERR_DEVICE_BAD_INDEX 8   /* reported by fme_read_device_status() */

/* Bits a kernel ORs into *dev_status. */
#define FME_DEV_TIMEOUT 0x1     /* a bounded wait inside a GEMM ran out; the kernel gave up */
#define FME_DEV_BAD_OFFSETS 0x2 /* offsets not rising from 0 to rows (or padded offsets invalid) */
#define FME_DEV_BAD_INDEX 0x4   /* an expert id or a gathered row index out of range */

#define FME_ROWWISE 0
#define FME_COLWISE 1
/* OR-ed into quantize_mxfp8's axis: the round-up scale variant (see there). */
#define FME_MX_SCALE_CEIL 0x100

#define FME_MAX_GROUPS 1024

/*
 * quantize_nvfp4_pertoken -- the NVFP4 variant of the MoE forward.
 *
 * Per row t of x [rows x k] (bf16): amax_t = max |x|, S_t = amax_t / 2688 (fp32,
 * IEEE correctly rounded division), per block b of 16: sb = E4M3(amax_b /
 * fl32(6 S_t)) (IEEE division), e = fl32(dec(sb) S_t), q = E2M1(x / e) (IEEE
 * division), round to nearest even, saturating.  A row with amax 0 or a block
 * whose scale code is 0 gets codes 0.  Rows are independent: a token's outputs
 * do not depend on any other row.
 *
 * Passage: "Composer 2 Technical Report" (papercache.org summary), section 6.1,
 * the NVFP4-variant paragraph (E2M1 values, an E4M3 scale per 16-element block,
 * an FP32 scale per token) and the hardware-math paragraph (IEEE-compliant
 * division when quantizing to this format); "Cursor Composer 2 report deep dive",
 * section 1 (per-token scales: no batch variance, no leakage from later tokens).
 *
 *   x          device bf16 [rows x k]
 *   rows, k    rows >= 0; k a multiple of 64, 64 <= k <= 8192
 *   offsets    device int32 [num_groups + 1] or NULL (see "Grouped rows");
 *              the groups only decide the padding of the scale layout
 *   num_groups 1 .. FME_MAX_GROUPS
 *   codes      device uint8 [rows x k/2]; element 2j in the low nibble of byte j
 *   sf         device uint8, fme_sf_bytes(rows, k, 16, num_groups) bytes, E4M3
 *   row_scale  device float [rows], S_t
 *   dev_status device int32 or NULL
 *   stream     cudaStream_t
 */
fme_status quantize_nvfp4_pertoken(const void *x, int64_t rows, int64_t k, const int32_t *offsets,
                                   int32_t num_groups, uint8_t *codes, uint8_t *sf, float *row_scale,
                                   int32_t *dev_status, void *stream);

/*
 * quantize_nvfp4_pertensor -- standard NVFP4, the comparator of the per-token
 * variant: the same steps with one FP32 scale for the whole tensor, S =
 * fl32(amax_x / 2688) where amax_x = max |x| over every row ("Cursor Composer 2
 * report deep dive", section 1, and "Composer 2 Technical Report", section 6.1:
 * standard NVFP4 scales per tensor, which makes a token's codes depend on the rest
 * of the batch).  Arguments as quantize_nvfp4_pertoken; row_scale[t] = S for
 * every row, so grouped_gemm_fwd_nvfp4 consumes the outputs unchanged.
 *   tensor_amax  device float [1], overwritten with amax_x (it is zeroed and
 *                reduced into on the stream first)
 */
fme_status quantize_nvfp4_pertensor(const void *x, int64_t rows, int64_t k, const int32_t *offsets,
                                    int32_t num_groups, uint8_t *codes, uint8_t *sf, float *row_scale,
                                    float *tensor_amax, int32_t *dev_status, void *stream);

/*
 * swiglu_quantize_nvfp4 -- the activation between the forward GEMMs fused with
 * the NVFP4 per-token quantization of its output.  Row t of gate_up [rows x
 * 2*inter] (bf16, the gate/up GEMM output) is [g (inter values) | u (inter
 * values)]; h = silu(g) * u, silu(v) = v / (1 + e^-v), evaluated in fp32 and
 * rounded to bf16 (nearest even), is quantized exactly as
 * quantize_nvfp4_pertoken quantizes a bf16 row (same codes, scale layout and row
 * scale for the same h).  The pages give DeepSeek-V3-class experts ("Scaling
 * and Optimizing Frontier Model Training", "MXFP8 expert kernels"); the gated
 * activation is their SwiGLU.
 *
 *   gate_up    device bf16 [rows x 2*inter]
 *   rows, inter  inter a multiple of 64, 64 <= inter <= 8192
 *   offsets, num_groups  as quantize_nvfp4_pertoken
 *   codes, sf, row_scale as quantize_nvfp4_pertoken with k = inter
 *   h          device bf16 [rows x inter] receiving the activation (needed by
 *              the backward), or NULL
 */
fme_status swiglu_quantize_nvfp4(const void *gate_up, int64_t rows, int64_t inter, const int32_t *offsets,
                                 int32_t num_groups, uint8_t *codes, uint8_t *sf, float *row_scale, void *h,
                                 int32_t *dev_status, void *stream);

/*
 * Routing: grouping the routed tokens by expert, and combining back.
 *
 * "Cursor Composer 2 report deep dive", section 2, and "Composer 2 Technical
 * Report" (papercache.org summary), section 6.1: tokens are quantized before they
 * are dispatched to their experts, and the experts' outputs are combined per token
 * in BF16.  Section 6.2 of the report: the expert choices per token are replayed
 * from the inference engine, so the grouping is a function of those ids alone.
 * Assignment a = t * top_k + k is token t's k-th expert, topk_ids[a].
 *
 * moe_route -- stable counting sort of the assignments by expert: offsets[E+1]
 * (rows per expert, prefix sums), row_of[a] = the grouped row of assignment a,
 * src_row[r] = the assignment of grouped row r.  Within an expert, rows follow a:
 * the grouping depends on the ids alone.  Ids outside [0, num_experts) get
 * row_of = -1, no grouped row, and FME_DEV_BAD_INDEX.
 *   topk_ids   device int32 [tokens x top_k]
 *   top_k      1 .. 64; num_experts 1 .. FME_MAX_GROUPS
 *   offsets    device int32 [num_experts + 1]
 *   row_of, src_row  device int32 [tokens x top_k]
 *   workspace  device scratch, fme_route_workspace_bytes(tokens, top_k, num_experts)
 *              bytes (16-byte aligned), contents irrelevant before and after
 */
fme_status moe_route(const int32_t *topk_ids, int64_t tokens, int32_t top_k, int32_t num_experts, int32_t *offsets,
                     int32_t *row_of, int32_t *src_row, void *workspace, int64_t workspace_bytes,
                     int32_t *dev_status, void *stream);

/*
 * moe_route_noalloc -- moe_route without a workspace argument and without any
 * allocation: the per-(chunk, expert) counters live in a static device array of
 * FME_ROUTE_STATIC_WORDS int32 inside the library, so
 * ceil(tokens * top_k / 1024) * num_experts must not exceed it
 * (FME_ERR_UNSUPPORTED_SHAPE otherwise).  Same outputs, bit for bit, as
 * moe_route.  Calls share that array: they must be ordered on the device (one
 * stream, or streams joined by events), never concurrent.  The array is part of
 * the library's device code: it is created when that code is loaded on a
 * device, which under CUDA's lazy module loading is the first call into
 * libfme.so on that device (any call).  Make that first call before relying on
 * the no-allocation property; the array then lives until the process exits.
 */
#define FME_ROUTE_STATIC_WORDS (1 << 20)
fme_status moe_route_noalloc(const int32_t *topk_ids, int64_t tokens, int32_t top_k, int32_t num_experts,
                             int32_t *offsets, int32_t *row_of, int32_t *src_row, int32_t *dev_status,
                             void *stream);

/*
 * permute_quantize_nvfp4 -- quantize_nvfp4_pertoken of the grouped token rows
 * X_g[r] = x[src_row[r] / top_k] without materialising X_g: codes, tiled scales
 * (padded per expert with these offsets) and row scales of the tokens in grouped
 * order, ready for grouped_gemm_fwd_nvfp4.  Gathered indices outside [0, tokens)
 * are reported (FME_DEV_BAD_INDEX).
 *   x          device bf16 [tokens x k]; k as quantize_nvfp4_pertoken
 *   src_row, offsets  from moe_route; the grouped rows are tokens * top_k
 */
fme_status permute_quantize_nvfp4(const void *x, int64_t tokens, int64_t k, const int32_t *src_row, int32_t top_k,
                                  const int32_t *offsets, int32_t num_experts, uint8_t *codes, uint8_t *sf,
                                  float *row_scale, int32_t *dev_status, void *stream);

/*
 * permute_quantize_mxfp8 -- quantize_mxfp8 row-wise of the grouped token rows
 * X_g[r] = x[src_row[r] / top_k]: MXFP8 codes [tokens*top_k x k] in grouped order
 * and their tiled scales (each expert padded to 128 rows), the quantize-before-
 * dispatch form of the grouped tokens.  Gathered indices outside [0, tokens) are
 * reported (FME_DEV_BAD_INDEX).
 *   x          device bf16 [tokens x k]; k a multiple of 32
 *   src_row, offsets  from moe_route
 */
fme_status permute_quantize_mxfp8(const void *x, int64_t tokens, int64_t k, const int32_t *src_row, int32_t top_k,
                                  const int32_t *offsets, int32_t num_experts, uint8_t *codes, uint8_t *sf,
                                  int32_t *dev_status, void *stream);

/*
 * moe_combine -- out[t, :] = bf16( sum_k weights[t, k] * y[row_of[t, k], :] ), the
 * sum over k in order in fp32, every product and every sum rounded to nearest
 * even (no fused multiply-add); assignments with row_of < 0 contribute nothing.
 *   y          device bf16 [rows_y x n], the grouped expert outputs
 *   row_of     from moe_route; weights device float [tokens x top_k]
 *   n          a multiple of 8
 *   out        device bf16 [tokens x n]
 */
fme_status moe_combine(const void *y, int64_t rows_y, const int32_t *row_of, const float *weights, int64_t tokens,
                       int32_t top_k, int64_t n, void *out, int32_t *dev_status, void *stream);

/*
 * quantize_mxfp8 -- standard MXFP8 (OCP MX v1.0 rule) of the MoE backward.
 *
 * Per block of 32: X = 2^(floor(log2 amax) - 8) stored as the E8M0 code
 * clamp(floor(log2 amax) + 119, 0, 254) (code 0 for an all-zero block);
 * q = E4M3(x / X), round to nearest even, saturating at 448.  X is a power of
 * two, so x / X is exact and the fast division the pages allow for MXFP8 gives
 * the same codes.
 *
 * Passage: "Composer 2 Technical Report", section 6.1, the MXFP8 paragraph of the
 * MoE backward (E4M3 values, an E8M0 scale per 32 elements) and the hardware-math
 * paragraph (a fast divide is acceptable for MXFP8); "Scaling and Optimizing
 * Frontier Model Training", "MXFP8 expert kernels".  The column-wise layout (blocks
 * along tokens, restarted at each expert) feeds the weight gradient.
 *
 * axis | FME_MX_SCALE_CEIL: the round-up scale variant, X = 2^ceil(log2(amax /
 * 448)) (code clamp(ceil(log2(amax / 448)) + 127, 0, 254)), the smallest power of
 * two that keeps every |x / X| <= 448, so no element saturates.  Layouts as below.
 *
 * axis = FME_ROWWISE: blocks run along each row of x [rows x cols].
 *   cols a multiple of 32, 32 <= cols <= 65536.
 *   codes  device uint8 [rows x cols] (E4M3)
 *   sf     device uint8, fme_sf_bytes(rows, cols, 32, num_groups) bytes (E8M0)
 *   padded_offsets must be NULL.
 *
 * axis = FME_COLWISE: blocks run down the columns, over the rows of one group at
 * a time.  Group g's rows are placed at padded positions starting at
 * P_g = 128 * sum_{g'<g} ceil(n_g'/128) and zero-filled up to the next multiple
 * of 128; blocks of 32 start at P_g.  The output is transposed so that the
 * position axis is contiguous:
 *   cols a multiple of 128.
 *   codes  device uint8 [cols x ld], ld = fme_colwise_ld(rows, num_groups);
 *          positions P_G .. ld-1 are left unwritten
 *   sf     device uint8, fme_sf_bytes(cols, ld, 32, 1) bytes: the scale matrix
 *          [cols x ld/32] in the tiled layout (rows = columns of x)
 *   padded_offsets device int32 [num_groups + 1]: P_0 .. P_G
 */
fme_status quantize_mxfp8(const void *x, int64_t rows, int64_t cols, int32_t axis, const int32_t *offsets,
                          int32_t num_groups, uint8_t *codes, uint8_t *sf, int32_t *padded_offsets,
                          int32_t *dev_status, void *stream);

/*
 * quantize_mxfp8_rowcol -- quantize_mxfp8 ROWWISE and COLWISE of the same x in one
 * pass (x is read once), e.g. dY of the backward, which feeds both dgrad
 * (row-wise) and wgrad (column-wise).  Outputs are identical, byte for byte, to
 * the two separate calls (cols a multiple of 128):
 *   row_codes, row_sf   as quantize_mxfp8(ROWWISE) with these offsets
 *   col_codes, col_sf   as quantize_mxfp8(COLWISE): [cols x ld], tiled scales
 *   padded_offsets      as quantize_mxfp8(COLWISE)
 * Row-wise scale bytes of padding rows are written as 0.
 */
fme_status quantize_mxfp8_rowcol(const void *x, int64_t rows, int64_t cols, const int32_t *offsets,
                                 int32_t num_groups, uint8_t *row_codes, uint8_t *row_sf, uint8_t *col_codes,
                                 uint8_t *col_sf, int32_t *padded_offsets, int32_t *dev_status, void *stream);

/*
 * swiglu_backward_quantize_mxfp8 -- the gate/up side of the expert backward.  With
 * the forward's h = silu(g) * u of the gate/up output [g | u] (silu(v) = v sigma(v),
 * "Scaling and Optimizing Frontier Model Training", "MXFP8 expert kernels": the
 * DeepSeek-V3-class experts; the activation read as SwiGLU) and dh the gradient of
 * h, computes d(gate/up) = [dg | du],
 *   dg = dh * u * sigma(g) * (1 + g * sigma(-g)),   du = dh * g * sigma(g),
 * in fp32, rounds it to bf16 and quantizes it as quantize_mxfp8_rowcol would
 * (row-wise for the gate/up dgrad, column-wise for its wgrad), in one pass.
 *   gate_up    device bf16 [rows x 2*inter]: [g | u] per row
 *   dh         device bf16 [rows x inter]
 *   inter      a multiple of 128, 128 .. 32768
 *   row_codes, row_sf, col_codes, col_sf, padded_offsets
 *              as quantize_mxfp8_rowcol of a [rows x 2*inter] tensor
 *   d_gate_up  device bf16 [rows x 2*inter] or NULL: the bf16 d(gate/up) that was
 *              quantized
 */
fme_status swiglu_backward_quantize_mxfp8(const void *gate_up, const void *dh, int64_t rows, int64_t inter,
                                          const int32_t *offsets, int32_t num_groups, uint8_t *row_codes,
                                          uint8_t *row_sf, uint8_t *col_codes, uint8_t *col_sf,
                                          int32_t *padded_offsets, void *d_gate_up, int32_t *dev_status,
                                          void *stream);

/*
 * grouped_gemm_fwd_nvfp4 -- Y[t, :] = S_x[t] * S_w[e, :] * sum_k A'[t,k] B'_e[:,k]
 * for every row t of expert e, where A', B' are the E2M1 codes times their E4M3
 * block scales, multiplied on the tensor cores with fp32 accumulation; the
 * epilogue applies (acc * S_x[t]) * S_w[e, n] in fp32 and rounds to bf16.
 * No split over K: a row's output does not depend on any other row.
 *
 * Passage: "Composer 2 Technical Report", section 6.1, the NVFP4-variant paragraph
 * (the per-token scale applied at the cost of GEMM-epilogue latency) and the
 * block-scaled tensor-core MMA sentence (dequantization inside the
 * systolic-array multiply); "Scaling and Optimizing Frontier Model Training",
 * "MXFP8 expert kernels" (grouped GEMMs over the experts' routed tokens).
 *
 *   a_codes, a_sf, a_scale  quantize_nvfp4_pertoken of X [m x k] with these offsets
 *   b_codes, b_sf, b_scale  quantize_nvfp4_pertoken of W [num_experts * n x k] as
 *                           one group (offsets NULL): expert e's rows are
 *                           e*n .. e*n+n-1, its scales the tiled layout's
 *                           128-row blocks e*n/128 ..
 *   offsets        device int32 [num_experts + 1], rows of X per expert
 *   m, n, k        n a multiple of 256; k a multiple of 256
 *   y              device bf16 [m x n]
 */
fme_status grouped_gemm_fwd_nvfp4(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_scale,
                                  const uint8_t *b_codes, const uint8_t *b_sf, const float *b_scale,
                                  const int32_t *offsets, int32_t num_experts, int64_t m, int64_t n,
                                  int64_t k, void *y, int32_t *dev_status, void *stream);

/*
 * grouped_gemm_fwd_nvfp4_swiglu -- the NVFP4 forward of the gate/up projection with
 * the activation in the epilogue: for every row t of expert e and every column j
 * of the intermediate width I = n / 2,
 *   g = S_x[t] * S_w[e, j]     * sum_k A'[t,k] B'_e[j, k]        (gate)
 *   u = S_x[t] * S_w[e, I + j] * sum_k A'[t,k] B'_e[I + j, k]    (up)
 *   h[t, j] = silu(g) * u,  silu(v) = v / (1 + e^-v),
 * g and u as grouped_gemm_fwd_nvfp4 forms them in fp32 before its bf16 rounding
 * (not rounded here), h evaluated in fp32 with a fast exponential and reciprocal
 * (relative error a few 2^-17) and rounded to bf16.  h then goes to
 * quantize_nvfp4_pertoken for the down projection: its per-token scale needs the
 * whole row of h, which no single output tile holds.
 *
 * Passages: as grouped_gemm_fwd_nvfp4 ("Composer 2 Technical Report", section 6.1,
 * the NVFP4-variant paragraph and the block-scaled MMA sentence).  The pages name
 * the gate/up projection but not its activation; SwiGLU with the gate in the
 * first n / 2 rows of each expert's W and the up projection in the last n / 2 is
 * this library's reading (the same as swiglu_quantize_nvfp4's [g | u] rows).
 *
 *   a_codes, a_sf, a_scale  quantize_nvfp4_pertoken of X [m x k] with these offsets
 *   b_codes, b_sf, b_scale  quantize_nvfp4_pertoken of W_gu [num_experts * n x k] as
 *                           one group: expert e's gate rows e*n .. e*n+I-1, its up
 *                           rows e*n+I .. e*n+n-1
 *   offsets        device int32 [num_experts + 1], rows of X per expert
 *   m, n, k        n (= 2 I) a multiple of 256; k a multiple of 256
 *   h              device bf16 [m x n / 2]
 * Errors and status words as grouped_gemm_fwd_nvfp4.
 */
fme_status grouped_gemm_fwd_nvfp4_swiglu(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_scale,
                                         const uint8_t *b_codes, const uint8_t *b_sf, const float *b_scale,
                                         const int32_t *offsets, int32_t num_experts, int64_t m, int64_t n,
                                         int64_t k, void *h, int32_t *dev_status, void *stream);

/*
 * grouped_gemm_fwd_mxfp8 -- the MXFP8 forward: Y[t, :] = sum_k A'[t,k] B'_e[:,k] for
 * every row t of expert e, A', B' = E4M3 codes times E8M0 block scales (blocks of
 * 32 along K), fp32 accumulation on the tensor cores, bf16 out; no per-token scale.
 * ("Scaling and Optimizing Frontier Model Training", "MXFP8 expert kernels": MXFP8
 * grouped GEMMs for the forward and backward of the expert layers.)
 *
 *   a_codes, a_sf  quantize_mxfp8(ROWWISE) of X [m x k] with these offsets
 *   b_codes, b_sf  quantize_mxfp8(ROWWISE) of W [num_experts * n x k], one group
 *                  (expert e's rows are e*n .. e*n+n-1)
 *   offsets        device int32 [num_experts + 1], rows of X per expert
 *   m, n, k        n a multiple of 256; k a multiple of 128
 *   y              device bf16 [m x n]
 */
fme_status grouped_gemm_fwd_mxfp8(const uint8_t *a_codes, const uint8_t *a_sf, const uint8_t *b_codes,
                                  const uint8_t *b_sf, const int32_t *offsets, int32_t num_experts, int64_t m,
                                  int64_t n, int64_t k, void *y, int32_t *dev_status, void *stream);

/*
 * grouped_gemm_dgrad_mxfp8 -- Y[t, :] = sum_j A'[t, j] B'[:, e*k + j] for every
 * row t of expert e (A', B' = E4M3 codes times E8M0 block scales), fp32
 * accumulation, bf16 out.  This is the data gradient dX_e = dY_e W_e when A is
 * the row-wise MXFP8 of dY [m x k] and B the column-wise MXFP8 of the stacked
 * weights W [num_experts * k x n] (one group), whose codes are [n x ldb].
 *
 * Passage: "Composer 2 Technical Report", section 6.1, the MXFP8 paragraph of the
 * MoE backward; "Scaling and Optimizing Frontier Model Training", "MXFP8 expert
 * kernels" (MXFP8 grouped GEMMs in the expert layers' backward).
 *
 *   a_codes, a_sf  quantize_mxfp8(ROWWISE) of A [m x k] with these offsets
 *   b_codes, b_sf  codes [n x ldb] and their scales (tiled, rows = n); expert e
 *                  uses columns e*k .. e*k+k-1, so ldb >= num_experts * k
 *   offsets        device int32 [num_experts + 1]
 *   m, n, k        n a multiple of 256; k a multiple of 128; ldb a multiple of 128
 *   y              device bf16 [m x n]
 */
fme_status grouped_gemm_dgrad_mxfp8(const uint8_t *a_codes, const uint8_t *a_sf, const uint8_t *b_codes,
                                    const uint8_t *b_sf, int64_t ldb, const int32_t *offsets,
                                    int32_t num_experts, int64_t m, int64_t n, int64_t k, void *y,
                                    int32_t *dev_status, void *stream);

/*
 * grouped_gemm_wgrad_mxfp8 -- Y_e[i, j] = sum_p A'[i, p] B'[j, p] over the padded
 * positions p of expert e, [P_e, P_e+1), fp32 accumulation over all of them (no
 * split), bf16 out.  With A = column-wise MXFP8 of dY and B = column-wise MXFP8
 * of H (same offsets) this is the weight gradient dW_e = dY_e^T H_e.  An
 * expert with no rows gets an all-zero Y_e.
 *
 * Passage: "Composer 2 Technical Report", section 6.1, the MXFP8 paragraph of the
 * MoE backward; "Scaling and Optimizing Frontier Model Training", "MXFP8 expert
 * kernels" (MXFP8 grouped GEMMs in the expert layers' backward).
 *
 *   a_codes, a_sf, lda  quantize_mxfp8(COLWISE) of dY [rows x m]: codes [m x lda]
 *   b_codes, b_sf, ldb  quantize_mxfp8(COLWISE) of H [rows x n]:  codes [n x ldb]
 *   padded_offsets  device int32 [num_experts + 1] written by those calls
 *   m, n            m and n multiples of 256, at most 65536
 *   y               device bf16 [num_experts x m x n]
 */
fme_status grouped_gemm_wgrad_mxfp8(const uint8_t *a_codes, const uint8_t *a_sf, int64_t lda,
                                    const uint8_t *b_codes, const uint8_t *b_sf, int64_t ldb,
                                    const int32_t *padded_offsets, int32_t num_experts, int64_t m,
                                    int64_t n, void *y, int32_t *dev_status, void *stream);

/*
 * grouped_gemm_wgrad_mxfp8_accumulate -- the same weight gradient added into an
 * fp32 buffer instead of written as bf16 (gradient accumulation over
 * micro-batches): dw_acc[e, i, j] = fl32(dw_acc[e, i, j] + Y_e[i, j]), one unfused
 * fp32 add per element, Y_e the fp32 accumulator of grouped_gemm_wgrad_mxfp8
 * (that call's bf16 output is Y_e rounded to bf16).  Experts with no rows leave
 * their dw_acc block untouched.  Arguments as grouped_gemm_wgrad_mxfp8, with
 *   dw_acc   device float [num_experts x m x n], read and written
 */
fme_status grouped_gemm_wgrad_mxfp8_accumulate(const uint8_t *a_codes, const uint8_t *a_sf, int64_t lda,
                                               const uint8_t *b_codes, const uint8_t *b_sf, int64_t ldb,
                                               const int32_t *padded_offsets, int32_t num_experts, int64_t m,
                                               int64_t n, float *dw_acc, int32_t *dev_status, void *stream);

/* Rows of the padded scale layout for `rows` rows in `num_groups` groups: an
 * upper bound of 128 * sum ceil(n_g / 128) that needs no offsets. */
int64_t fme_sf_padded_rows(int64_t rows, int32_t num_groups);

/* Bytes of a tiled scale buffer for a [rows x cols] tensor quantized in blocks
 * of `block` (16 or 32) along cols, in `num_groups` groups. */
int64_t fme_sf_bytes(int64_t rows, int64_t cols, int32_t block, int32_t num_groups);

/* Leading dimension (positions per column) of the column-wise MXFP8 outputs. */
int64_t fme_colwise_ld(int64_t rows, int32_t num_groups);

/* Bytes of moe_route's workspace (at least 16). */
int64_t fme_route_workspace_bytes(int64_t tokens, int32_t top_k, int32_t num_experts);

/* Synchronises `stream`, copies *dev_status to the host and maps it to a status,
 * the first of these whose bit is set: FME_ERR_DEVICE_BAD_OFFSETS,
 * FME_ERR_DEVICE_BAD_INDEX, FME_ERR_DEVICE_TIMEOUT; FME_OK when none is.  `raw`
 * (may be NULL) receives the raw bits. */
fme_status fme_read_device_status(const int32_t *dev_status, void *stream, int32_t *raw);

/* Static text for a status code. */
const char *fme_error_string(fme_status status);

/* Text of the last CUDA error seen by a call on this thread ("" if none). */
const char *fme_last_cuda_error(void);

/* Library version string. */
const char *fme_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FME_H */

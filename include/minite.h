/*
 * minite.h -- C ABI of the native-NVFP4 W4A4 MoE expert MLP (GB300, sm_103a).
 *
 * The path: per-token NVFP4 quantization fused into the MoE permutation and
 * into the routing-weighted SwiGLU, a block-scaled grouped GEMM over experts
 * that reads contiguous expert buffers and device-side offsets, and the
 * combine back to token order.
 *
 * Sources. "miniTE Technical Report: Stable and Efficient Reinforcement
 * Learning with Native NVFP4" (summary page), section "Follow the numerical
 * execution path" (per-token activation scaling) and section "Two
 * complementary interventions" (amax computed during permutation and during
 * weighted SwiGLU; scale-layout conversion fused with quantization;
 * contiguous buffers with device-side metadata). "miniTE accélère le RL en
 * NVFP4 sur B300", lead (W4A4) and section "Diagnostic, alignement et noyaux
 * rapides" (grouped GEMMs over the experts of a MoE layer).
 *
 * Common rules for every entry point:
 *  - Pointers named *device* are CUDA device pointers owned by the caller.
 *    The library allocates no memory and keeps no pointer after a call
 *    returns. Buffers must not overlap unless stated.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *    never synchronizes the host. Host-detectable errors (null pointers, bad
 *    shapes, bad alignment) are returned before anything is enqueued.
 *  - Errors found on the device (routing ids out of range, a pipeline wait
 *    that timed out) are OR-ed as bits (1 << code) into `*status`, a caller
 *    owned device int32 that the caller zeroes and reads after its own
 *    synchronization. `status` may be NULL, in which case they are dropped.
 *  - BF16 tensors are raw 16-bit patterns (`const void*`), row-major.
 *  - NVFP4 data: codes are packed E2M1, two per byte, element 2i in the low
 *    nibble; scale factors (SF) are unsigned E4M3 bytes, one per 16 elements
 *    along the blocked dimension, stored in 128-row x 4-column atoms of
 *    512 bytes: for a region with rows padded to 128 and Kc = roundup(K/16, 4)
 *    SF columns, the SF of row r, column c is at byte
 *      ((r/128)*(Kc/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4.
 *    Padding bytes are written as 0. Dequantized value = e2m1(code) * sf / g.
 *  - Global scale g (FP32): 2688 / amax of the row (activations) or of the
 *    whole group (weights), capped at FLT_MAX; 1 when amax is 0.
 *  - Base pointers must be 16-byte aligned; the GEMM operands 128-byte.
 */
#ifndef MINITE_H
#define MINITE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* minite_stream_t;

typedef enum {
  MINITE_OK = 0,
  MINITE_ERR_INVALID_ARG = 1,      /* null pointer, bad enum, bad alignment, small workspace */
  MINITE_ERR_UNSUPPORTED_SHAPE = 2,/* a size rule below is violated */
  MINITE_ERR_CUDA = 3,             /* a CUDA launch or runtime call failed */
  MINITE_ERR_TIMEOUT = 4,          /* device: a pipeline wait gave up (status bit 1<<4) */
  MINITE_ERR_BAD_ROUTING = 5,      /* device: a routing id outside [0, E) (status bit 1<<5) */
  MINITE_ERR_SCRATCH_LIMIT = 6     /* the problem needs more scratch than the built-in array */
} minite_status_t;

enum { MINITE_SCALE_PER_ROW = 0, MINITE_SCALE_PER_GROUP = 1 };
enum { MINITE_ALONG_COLS = 0, MINITE_ALONG_ROWS = 1 };
enum { MINITE_OUT_BF16 = 0, MINITE_OUT_FP32 = 1 };
enum {
  MINITE_OP_QUANTIZE = 0,
  MINITE_OP_PERMUTE_QUANT = 1,
  MINITE_OP_COMBINE_BACKWARD_QUANT = 2,
  MINITE_OP_QUANTIZE_TOKENS = 3,
  MINITE_OP_GATE_UP_SWIGLU = 4
};

/*
 * minite_quantize_nvfp4 -- NVFP4 quantization of `groups` BF16 matrices.
 *
 * Cites: per-token activation scaling ("Follow the numerical execution
 * path"); swizzled scale layout written by the quantizer itself ("Two
 * complementary interventions").
 *
 * x:           device, BF16 [groups, rows, cols], 16-byte aligned (32-byte
 *              aligned x is read with 32-byte loads).
 * scale_mode:  MINITE_SCALE_PER_ROW: one g per quantized row (activations);
 *              MINITE_SCALE_PER_GROUP: one g per group from the amax of the
 *              whole group (one expert's weight matrix).
 * orientation: MINITE_ALONG_COLS: blocks of 16 along cols; the quantized
 *              matrix of a group is x[g] itself, [rows, cols].
 *              MINITE_ALONG_ROWS: blocks of 16 along rows; the quantized
 *              matrix is x[g] transposed, [cols, rows] (the dgrad layout of a
 *              forward weight).
 *              Let (Rq, Cq) be the quantized matrix's shape: (rows, cols) or
 *              (cols, rows).
 * gscale_in:   device float [groups] or NULL. PER_GROUP only: use these g
 *              instead of computing the amax (re-quantizing a weight in the
 *              other orientation with the same global scale).
 * codes:       device, uint8 [groups, Rq, Cq/2], 8-byte aligned.
 * sf:          device, uint8 [groups, roundup(Rq,128) * roundup(Cq/16,4)],
 *              4-byte aligned.
 * gscale_out:  device float, [groups*Rq] (PER_ROW) or [groups] (PER_GROUP).
 *              May equal gscale_in.
 * workspace:   device, >= minite_workspace_bytes(MINITE_OP_QUANTIZE, groups,
 *              0, 0, 0) bytes (PER_GROUP without gscale_in only; else NULL ok).
 * Shape rules: Cq % 16 == 0 (blocks), cols % 8 == 0, all > 0; ALONG_COLS:
 * cols <= 4096; ALONG_ROWS: PER_GROUP only, rows, cols < 2^30; PER_GROUP: rows * cols / 16 <
 * 2^32; groups * rows * cols < 2^40. Misaligned pointers: INVALID_ARG;
 * other shapes: UNSUPPORTED_SHAPE (nothing enqueued in either case).
 */
int minite_quantize_nvfp4(const void* x, int64_t groups, int64_t rows, int64_t cols,
                          int scale_mode, int orientation, const float* gscale_in,
                          uint8_t* codes, uint8_t* sf, float* gscale_out,
                          void* workspace, size_t ws_bytes, int32_t* status,
                          minite_stream_t stream);

/*
 * minite_quantize_nvfp4_dual -- per-group (weight) NVFP4 quantization in both
 * orientations from one read of x: the forward copy with blocks of 16 along
 * cols and the dgrad copy (x[g] transposed) with blocks of 16 along rows,
 * both with the group's global scale g = 2688 / amax(x[g]).
 *
 * Cites: the weight recipe of "Follow the numerical execution path"
 * (per-tensor FP32 global scale, E4M3 block scales) and the fused scale
 * layout of "Two complementary interventions". The pages do not describe a
 * two-orientation pass; the results are exactly those of
 * minite_quantize_nvfp4(PER_GROUP, ALONG_COLS) followed by
 * minite_quantize_nvfp4(PER_GROUP, ALONG_ROWS, gscale_in = its g).
 *
 * x:          device, BF16 [groups, rows, cols], 16-byte aligned.
 * codes_k:    device, uint8 [groups, rows, cols/2], 8-byte aligned.
 * sf_k:       device, uint8 [groups, roundup(rows,128) * roundup(cols/16,4)].
 * codes_n:    device, uint8 [groups, cols, rows/2], 8-byte aligned.
 * sf_n:       device, uint8 [groups, roundup(cols,128) * roundup(rows/16,4)].
 * gscale_out: device float [groups].
 * workspace:  device, >= minite_workspace_bytes(MINITE_OP_QUANTIZE, groups,
 *             0, 0, 0) bytes; contents on entry are ignored.
 * Shape rules: rows % 16 == 0, cols % 16 == 0, rows, cols < 2^30,
 * groups * rows * cols < 2^40.
 */
int minite_quantize_nvfp4_dual(const void* x, int64_t groups, int64_t rows, int64_t cols,
                               uint8_t* codes_k, uint8_t* sf_k, uint8_t* codes_n,
                               uint8_t* sf_n, float* gscale_out, void* workspace,
                               size_t ws_bytes, int32_t* status, minite_stream_t stream);

/*
 * minite_moe_permute_quant -- MoE permutation fused with per-token amax,
 * NVFP4 quantization and the SF swizzle, in one pass over x.
 *
 * Cites: "Two complementary interventions" (amax during permutation,
 * contiguous buffers, device-side metadata, fused scale layout) and "Follow
 * the numerical execution path" (per-token scales).
 *
 * Permuted rows are ordered by (expert, token, slot). Row p holds the
 * quantization of token perm_src[p]; a token routed to k experts appears in
 * k rows with identical codes, SF and g. Pairs with an id outside [0, E) are
 * dropped (status bit 1<<MINITE_ERR_BAD_ROUTING, dest_row = -1), so the used
 * rows are [0, expert_offsets[E]) and later rows are left untouched.
 *
 * x:              device, BF16 [T, H].
 * topk_ids:       device, int32 [T, k].
 * topk_w:         device, float [T, k], or NULL (then perm_w must be NULL).
 * codes:          device, uint8 [T*k, H/2].
 * sf:             device, uint8 [(T*k + 128*E) * roundup(H/16,4)]. Expert e's
 *                 rows occupy the padded row range [sf_row_offsets[e],
 *                 sf_row_offsets[e+1]) (local row = p - expert_offsets[e]).
 * row_g:          device, float [T*k].
 * expert_offsets: device, int32 [E+1], exclusive prefix of expert counts.
 * sf_row_offsets: device, int32 [E+1], prefix of counts rounded up to 128.
 * perm_src:       device, int32 [T*k], token of each permuted row.
 * dest_row:       device, int32 [T, k], permuted row of each (token, slot).
 * perm_w:         device, float [T*k], routing weight of each row, or NULL.
 * workspace:      device, >= minite_workspace_bytes(MINITE_OP_PERMUTE_QUANT,
 *                 T, H, E, k) bytes; contents on entry are ignored.
 * Shape rules: H % 64 == 0, 1 <= E <= 1024, 1 <= k <= 32, T >= 1,
 * T*k < 2^31.
 */
int minite_moe_permute_quant(const void* x, const int32_t* topk_ids, const float* topk_w,
                             int64_t T, int64_t H, int32_t E, int32_t k,
                             uint8_t* codes, uint8_t* sf, float* row_g,
                             int32_t* expert_offsets, int32_t* sf_row_offsets,
                             int32_t* perm_src, int32_t* dest_row, float* perm_w,
                             void* workspace, size_t ws_bytes, int32_t* status,
                             minite_stream_t stream);

/*
 * minite_moe_permute_quant_noalloc -- minite_moe_permute_quant for callers
 * that cannot allocate device memory. The sources describe no counterpart
 * to this entry point; it exists for deployment only.
 *
 * Same arguments, outputs and results as minite_moe_permute_quant, minus the
 * workspace: the scratch lives in a 2 MiB array inside the library's device
 * memory, held by every GPU that loads the library until the process exits.
 * Use it where calling cudaMalloc is not possible: a fixed memory plan, a
 * plugin that only receives its inputs and outputs, a loop that must not
 * enter the allocator. It allocates nothing and calls no allocating routine.
 *  - Limit: the ranking scratch must fit in the 2 MiB array. It takes
 *    4*E*ceil(T / floor(512/k)) bytes (one expert histogram per chunk of
 *    floor(512/k) tokens) plus 4*E + 256 bytes, each part rounded up to 256
 *    bytes (at k = 8 about T*E <= 32M). Larger problems return
 *    MINITE_ERR_SCRATCH_LIMIT before anything is enqueued.
 *    minite_workspace_bytes(MINITE_OP_PERMUTE_QUANT, ...) also counts the
 *    token-order staging of the scales; when that staging does not fit in
 *    the array as well, each token's scales are written straight to its k
 *    rows instead, with identical results.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *    The address is kept for the life of the process: after
 *    cudaDeviceReset the library's module is reloaded elsewhere, so do not
 *    call this entry point again in a process that reset its device.
 *  - All calls on a device share the array: calls that overlap on the GPU
 *    (different streams with no ordering between them) race. Nothing needs
 *    clearing between calls; every scratch word read is rewritten first.
 */
int minite_moe_permute_quant_noalloc(const void* x, const int32_t* topk_ids,
                                     const float* topk_w, int64_t T, int64_t H, int32_t E,
                                     int32_t k, uint8_t* codes, uint8_t* sf, float* row_g,
                                     int32_t* expert_offsets, int32_t* sf_row_offsets,
                                     int32_t* perm_src, int32_t* dest_row, float* perm_w,
                                     int32_t* status, minite_stream_t stream);

/*
 * minite_grouped_gemm_nvfp4 -- block-scaled FP4 x FP4 grouped GEMM over
 * experts, one launch for all experts.
 *
 * Cites: "Diagnostic, alignement et noyaux rapides" (grouped GEMMs for MoE);
 * "Two complementary interventions" (contiguous expert buffers, device-side
 * metadata: the host never learns the per-expert row counts).
 *
 * For every row m in [0, expert_offsets[E]) of expert e (offsets[e] <= m <
 * offsets[e+1]) and n in [0, N):
 *   out[m, n] = sum_k (a(m,k) * sfa(m,k/16)) * (b_e(n,k) * sfb_e(n,k/16))
 *               / (a_g[m] * b_g[e])
 * with a, b the E2M1 values; accumulation in FP32 on the tensor cores in a
 * fixed K order with no split-K, so a row's result depends only on its own
 * codes and its expert's weights.
 *
 * a_codes:  device, uint8 [M_total, K/2], rows in permuted order.
 * a_sf:     device, SF of A in per-expert padded regions (sf_row_offsets).
 * a_g:      device, float [M_total], per-row global scales.
 * b_codes:  device, uint8 [E, N, K/2] (K-major weights).
 * b_sf:     device, uint8 [E, roundup(N,128) * roundup(K/16,4)].
 * b_g:      device, float [E].
 * expert_offsets, sf_row_offsets: device, int32 [E+1] (as produced by
 *           minite_moe_permute_quant; for a dense GEMM {0, M} and
 *           {0, roundup(M,128)}).
 * M_total:  number of rows of a_codes / out (upper bound of offsets[E]).
 * out:      device, [M_total, N] BF16 (round to nearest even) or FP32; rows
 *           at or beyond offsets[E] are not written.
 * Shape rules: K % 64 == 0, N % 32 == 0, 1 <= E <= 1024, M_total < 2^31,
 * a_codes/b_codes 128-byte and out 32-byte aligned.
 */
int minite_grouped_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_g,
                              const uint8_t* b_codes, const uint8_t* b_sf, const float* b_g,
                              const int32_t* expert_offsets, const int32_t* sf_row_offsets,
                              int64_t M_total, int64_t N, int64_t K, int32_t E,
                              void* out, int out_dtype, int32_t* status,
                              minite_stream_t stream);

/*
 * minite_gate_up_swiglu_quant_nvfp4 -- the gate_up grouped GEMM with the
 * routing-weighted SwiGLU and the NVFP4 requantization of its result fused
 * into the GEMM's epilogue: the gate_up product never goes through memory
 * unless gate_up is given.
 *
 * Cites: "Two complementary interventions" (amax computed during weighted
 * SwiGLU, fused scale layout) and "Diagnostic, alignement et noyaux rapides"
 * (grouped GEMMs over experts).
 *
 * Bit for bit the composition
 *   minite_grouped_gemm_nvfp4(a..., b..., N = 2I, out = BF16 gate_up)
 *   minite_swiglu_weighted_quant(gate_up, perm_w, ...)
 * on the same arguments: each row's gate and up values are rounded to BF16
 * exactly as that GEMM stores them before the SwiGLU, and the row's global
 * scale comes from the |h| maximum over all I columns.
 *
 * a_codes, a_sf, a_g, b_codes, b_sf, b_g, expert_offsets, sf_row_offsets,
 * M_total, K, E: as for minite_grouped_gemm_nvfp4 with N = 2I (b_codes
 *          [E, 2I, K/2]: gate rows [0, I), up rows [I, 2I); b_g [E]).
 * perm_w:  device float [M_total] or NULL (weight 1).
 * gate_up: device BF16 [M_total, 2I], 32-byte aligned, or NULL: when given it
 *          also receives the GEMM's BF16 output (for a backward pass).
 * h_codes, h_sf, h_g: as the codes, sf and row_g of
 *          minite_swiglu_weighted_quant (16-byte aligned); padding rows of
 *          each expert's scale region are zeroed.
 * workspace: device, >= minite_workspace_bytes(MINITE_OP_GATE_UP_SWIGLU,
 *          M_total, I, 0, 0) bytes (4 * M_total * roundup(I/128, 4)),
 *          16-byte aligned; contents on entry are ignored (the call clears
 *          what it uses first).
 * Shape rules: I % 128 == 0, 128 <= I <= 8192, K % 64 == 0, 1 <= E <= 663
 * (the kernel's shared memory, 219.2 KB + 12 (E+1) bytes, within 227 KB),
 * M_total < 2^31; otherwise MINITE_ERR_UNSUPPORTED_SHAPE and nothing is
 * enqueued.
 * Device errors: invalid offsets set bit 1<<MINITE_ERR_INVALID_ARG; the
 * I/128 tiles of a 256-row block exchange their rows' maxima through the
 * workspace, and a wait for that exchange (like every other wait) gives up
 * after the budget of minite_set_wait_budget_ns with bit
 * 1<<MINITE_ERR_TIMEOUT. Calls sharing a workspace must not overlap.
 */
int minite_gate_up_swiglu_quant_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf,
                                      const float* a_g, const uint8_t* b_codes,
                                      const uint8_t* b_sf, const float* b_g,
                                      const int32_t* expert_offsets,
                                      const int32_t* sf_row_offsets, int64_t M_total, int64_t I,
                                      int64_t K, int32_t E, const float* perm_w, void* gate_up,
                                      uint8_t* h_codes, uint8_t* h_sf, float* h_g,
                                      void* workspace, size_t ws_bytes, int32_t* status,
                                      minite_stream_t stream);

/*
 * minite_grouped_gemm_wgrad_nvfp4 -- weight gradient of a grouped
 * projection, one launch for all experts, from two token-axis operands of
 * minite_quantize_tokens_nvfp4 over the same routing (same kofs):
 *   out[e, m, n] = sum_{k in [kofs[e], kofs[e+1])} (a(m,k) sfa(m,k/16))
 *                  * (b(n,k) sfb(n,k/16)) / (a_g[e] * b_g[e])
 * accumulated in FP32 on the tensor cores in a fixed K order (no split-K).
 * Experts without tokens are not written.
 *
 * Cites: "Diagnostic, alignement et noyaux rapides" (grouped GEMMs over
 * experts) and miniTE report summary, "Two complementary interventions"
 * (device-side per-expert metadata); the pages' backward is BF16, so this
 * NVFP4 weight gradient is a reading.
 *
 * a_codes: device, uint8 [M, k_cap/2], 128-byte aligned; a_sf: its scales
 *          (k_cap/16 scale columns), 16-byte aligned; a_g: device float [E].
 * b_codes, b_sf, b_g: the same for the N-channel operand.
 * kofs:    device, int32 [E+1]: 0, non-decreasing, multiples of 256, at most
 *          k_cap; otherwise nothing is written and bit 1<<MINITE_ERR_INVALID_ARG
 *          is set in *status.
 * out:     device, [E, M, N] BF16 or FP32 (out_dtype), 32-byte aligned.
 * Shape rules: 1 <= M <= 65536, N % 32 == 0, 32 <= N <= 65536,
 * k_cap % 256 == 0, 1 <= E <= 1024. Waits are bounded as in
 * minite_grouped_gemm_nvfp4.
 */
int minite_grouped_gemm_wgrad_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_g,
                                    const uint8_t* b_codes, const uint8_t* b_sf, const float* b_g,
                                    const int32_t* kofs, int32_t E, int64_t M, int64_t N,
                                    int64_t k_cap, void* out, int out_dtype, int32_t* status,
                                    minite_stream_t stream);

/*
 * minite_swiglu_weighted_quant -- routing-weighted SwiGLU with the per-row
 * amax and NVFP4 requantization fused into the same pass.
 *
 * Cites: "Two complementary interventions" (amax computed during weighted
 * SwiGLU, fused scale layout).
 *
 * For each used row m (< expert_offsets[E]):
 *   h = (silu(gate) * up) * w,  gate = gate_up[m, 0:I], up = gate_up[m, I:2I],
 *   silu(v) = v / (1 + exp(-v)), w = perm_w[m] (1 if perm_w is NULL),
 * all in FP32 with a specified exponential (Cody-Waite reduction, degree-7
 * Taylor polynomial, inputs clamped to [-87, 88]); then h is quantized per
 * row exactly as minite_quantize_nvfp4 PER_ROW, with the SF written into the
 * per-expert padded regions given by sf_row_offsets.
 *
 * gate_up: device, BF16 [M, 2I], 32-byte aligned.  perm_w: device float [M]
 *          or NULL.
 * codes:   device, uint8 [M, I/2], 16-byte aligned.  sf: as for the permute
 *          output with I in place of H, 16-byte aligned.  row_g: device,
 *          float [M].
 * Shape rules: I % 64 == 0, 64 <= I <= 2048, 1 <= E <= 1024, M < 2^31.
 */
int minite_swiglu_weighted_quant(const void* gate_up, const float* perm_w,
                                 int64_t M, int64_t I, int32_t E,
                                 const int32_t* expert_offsets, const int32_t* sf_row_offsets,
                                 uint8_t* codes, uint8_t* sf, float* row_g,
                                 int32_t* status, minite_stream_t stream);

/*
 * minite_swiglu_weighted_quant_keep_h -- minite_swiglu_weighted_quant that
 * also stores h (the FP32 values it quantizes, each rounded to BF16 to
 * nearest even) in h_out, device BF16 [M, I], 32-byte aligned, rows in
 * permuted order; rows at or beyond expert_offsets[E] are not written. h is
 * what the down projection's weight gradient needs from the forward (see
 * minite_quantize_tokens_nvfp4). h_amax, device float [M] or NULL: when
 * given, h_amax[m] = max |h_out[m, :]| for every row written (the row's FP32
 * maximum rounded to BF16, which is the maximum of the rounded row because
 * rounding is monotone), the per-row maxima that minite_quantize_tokens_nvfp4
 * takes instead of re-reading h: the maximum taken inside the pass that
 * produces the values, as the miniTE report summary's "Two complementary
 * interventions" does for the permutation and the weighted SwiGLU. Same
 * arguments, rules and errors otherwise; h_out may not be NULL.
 */
int minite_swiglu_weighted_quant_keep_h(const void* gate_up, const float* perm_w, int64_t M,
                                        int64_t I, int32_t E, const int32_t* expert_offsets,
                                        const int32_t* sf_row_offsets, uint8_t* codes,
                                        uint8_t* sf, float* row_g, void* h_out, float* h_amax,
                                        int32_t* status, minite_stream_t stream);

/*
 * minite_swiglu_backward_quant -- gradient of the routing-weighted SwiGLU
 * with respect to its gate and up inputs, with per-row NVFP4 requantization
 * of the result fused into the same pass (the A operand of the gate_up
 * dgrad GEMM).
 *
 * Cites: miniTE report summary, "Two complementary interventions" (amax
 * computed inside the SwiGLU pass, fused scale layout) and "Respect the
 * timing boundaries" (the backward of the learner's expert MLP; the pages
 * run it in BF16, this entry point is the NVFP4 variant of that step).
 *
 * For each used row m (< expert_offsets[E]), with g = gate_up[m, 0:I],
 * u = gate_up[m, I:2I], w = perm_w[m] (1 if perm_w is NULL) and the
 * gradient dh[m, 0:I] of h = (silu(g) * u) * w:
 *   d = 1 + exp(-g), s = 1 / d, silu = g / d, silu' = s * (1 + g * (1 - s))
 *   dg = ((dh * u) * w) * silu',  du = (dh * silu) * w
 * every step one FP32 operation rounded to nearest, in this order, with the
 * exponential of minite_swiglu_weighted_quant. The row [dg | du] (2I values)
 * is then quantized per row exactly as minite_quantize_nvfp4 PER_ROW, the SF
 * written into the per-expert padded regions given by sf_row_offsets; the
 * SF bytes of each expert's padding rows are set to 0.
 *
 * gate_up: device, BF16 [M, 2I], 32-byte aligned (the forward's gate_up
 *          GEMM output).  dh: device, BF16 [M, I], 32-byte aligned.
 * perm_w:  device float [M] or NULL.
 * codes:   device, uint8 [M, I] (2I E2M1 codes per row), 16-byte aligned.
 * sf:      device, uint8 [(M + 128 E) * (2I/16)] at most, 16-byte aligned,
 *          rows per expert as sf_row_offsets says.  row_g: device, float [M].
 * Rows at or beyond expert_offsets[E] are not written. Inconsistent offsets
 * make the kernel write nothing and store MINITE_ERR_INVALID_ARG in *status.
 * A row whose dg or du overflows FP32 (or holds NaN) has no finite amax;
 * its codes, scales and global scale are unspecified.
 * All buffers are owned by the caller; the call is asynchronous on stream.
 * Shape rules: I % 64 == 0, 64 <= I <= 2048, 1 <= E <= 1024, M < 2^31.
 */
int minite_swiglu_backward_quant(const void* gate_up, const void* dh, const float* perm_w,
                                 int64_t M, int64_t I, int32_t E,
                                 const int32_t* expert_offsets, const int32_t* sf_row_offsets,
                                 uint8_t* codes, uint8_t* sf, float* row_g,
                                 int32_t* status, minite_stream_t stream);

/*
 * minite_swiglu_backward_quant_keep -- minite_swiglu_backward_quant that also
 * stores [dg | du] (the FP32 values it quantizes, each rounded to BF16 to
 * nearest even) in dgu_out, device BF16 [M, 2I], 32-byte aligned, rows in
 * permuted order; rows at or beyond expert_offsets[E] are not written. The
 * gate_up projection's weight gradient takes its token-axis operand from it
 * (see minite_quantize_tokens_nvfp4). dgu_amax, device float [M] or NULL:
 * when given, dgu_amax[m] = max |dgu_out[m, :]| for every row written (as
 * h_amax of minite_swiglu_weighted_quant_keep_h). Same arguments, rules and
 * errors otherwise; dgu_out may not be NULL.
 */
int minite_swiglu_backward_quant_keep(const void* gate_up, const void* dh, const float* perm_w,
                                      int64_t M, int64_t I, int32_t E,
                                      const int32_t* expert_offsets, const int32_t* sf_row_offsets,
                                      uint8_t* codes, uint8_t* sf, float* row_g, void* dgu_out,
                                      float* dgu_amax, int32_t* status, minite_stream_t stream);

/*
 * minite_moe_combine -- unpermute: y[t] = BF16(sum_{j<k} D[dest_row[t,j]]),
 * summed in FP32 in slot order starting from 0; dropped pairs (dest_row < 0)
 * are skipped. The routing weight is already inside D (applied in the
 * SwiGLU).
 *
 * expert_out: device, BF16 [M, N], rows in permuted order.
 * dest_row:   device, int32 [T, k]; entries >= M are skipped and reported
 *             as status bit 1<<MINITE_ERR_BAD_ROUTING.
 * y:          device, BF16 [T, N]; must not overlap expert_out.
 * Shape rules: N % 8 == 0, 1 <= k <= 32.
 */
int minite_moe_combine(const void* expert_out, const int32_t* dest_row,
                       int64_t T, int64_t M, int64_t N, int32_t k, void* y,
                       int32_t* status, minite_stream_t stream);

/*
 * minite_moe_combine_backward_quant -- the backward of the combine with the
 * NVFP4 quantization of its result fused in: dD[dest_row[t, j]] = dY[t] for
 * every routed pair (t, j), i.e. dY laid out like the forward's permuted
 * activations, quantized per token exactly as minite_moe_permute_quant
 * quantizes x (same codes, scales, layout and row_g), reusing the forward
 * permutation's routing instead of ranking the routing ids again. The
 * result is the A operand of the down-projection dgrad GEMM.
 *
 * Cites: miniTE report summary, "Follow the numerical execution path"
 * (per-token scaling) and "Two complementary interventions" (contiguous
 * expert buffers, device-side metadata, fused scale layout), applied to the
 * backward; the pages run the backward in BF16 ("Respect the timing
 * boundaries"), so this NVFP4 variant is a reading.
 *
 * dy:        device, BF16 [T, H], 16-byte aligned.
 * dest_row, expert_offsets, sf_row_offsets, perm_src: device, the forward
 *            permutation's outputs for the same routing (unchanged).
 * codes, sf, row_g: device outputs as for minite_moe_permute_quant.
 * workspace: device, >= minite_workspace_bytes(MINITE_OP_COMBINE_BACKWARD_QUANT,
 *            T, H, 0, 0) bytes, 256-byte aligned, caller-owned scratch.
 * The routing is checked on the device: inconsistent offsets make the
 * kernels write nothing; a dest_row past expert_offsets[E] or a perm_src
 * outside [0, T) is skipped; each sets bit 1<<MINITE_ERR_INVALID_ARG in
 * *status. The call is asynchronous on stream.
 * Shape rules: as minite_moe_permute_quant.
 */
int minite_moe_combine_backward_quant(const void* dy, int64_t T, int64_t H, int32_t E, int32_t k,
                                      const int32_t* dest_row, const int32_t* expert_offsets,
                                      const int32_t* sf_row_offsets, const int32_t* perm_src,
                                      uint8_t* codes, uint8_t* sf, float* row_g,
                                      void* workspace, size_t ws_bytes, int32_t* status,
                                      minite_stream_t stream);

/*
 * minite_quantize_tokens_nvfp4 -- one operand of a weight-gradient GEMM:
 * each expert's permuted rows transposed to [channels, tokens] and quantized
 * in blocks of 16 consecutive tokens, one FP32 global scale per expert.
 *
 * Cites: miniTE report summary, "Two complementary interventions"
 * (contiguous expert buffers, device-side metadata, scale layout written by
 * the quantizer) and "Respect the timing boundaries" (the pages' backward is
 * BF16; quantizing the weight gradient's operands along tokens is a reading:
 * the gradient sums over the expert's tokens, so no scale may vary along
 * them).
 *
 * Permuted row m (expert e of the offsets) holds x[row_src[m]] (or x[m] when
 * row_src is NULL). For expert e with c_e rows, K range [kofs[e], kofs[e+1])
 * where kofs is the prefix of c_e rounded up to 256 (written to kofs_out):
 *   g[e] = min(2688 / amax(rows of e), FLT_MAX), 1 for amax 0;
 *   column kofs[e] + j of channel row c holds x_e[j, c] for j < c_e, 0 after,
 *   quantized as in minite_quantize_nvfp4 with blocks along the columns.
 *
 * x:         device, BF16 [x_rows, C], 16-byte aligned.
 * row_src:   device, int32 [m_cap] (e.g. perm_src of the permutation), or
 *            NULL (then rows are x's own and m_cap <= x_rows).
 * row_amax:  device, float [x_rows], or NULL. When given, row_amax[r] must
 *            be max_c |x[r, c]| (as the SwiGLU entries that keep their BF16
 *            output write it); the experts' maxima are then taken from it
 *            and x is read once (by the encoding) instead of twice. The
 *            results equal those of a NULL row_amax.
 * m_cap:     permuted rows available (>= expert_offsets[E]).
 * expert_offsets: device, int32 [E+1] (the permutation's).
 * k_cap:     token columns allocated, a multiple of 256 and >= kofs[E]
 *            (M + 256 E always suffices).
 * codes:     device, uint8 [C, k_cap / 2] (row pitch k_cap / 2), 32-byte
 *            aligned. sf: device, [roundup(C, 128) * k_cap / 16] bytes,
 *            128-row x 4-column atoms with k_cap / 16 scale columns; rows past
 *            C are zeroed up to column kofs[E] / 16.
 * g_out:     device, float [E]. kofs_out: device, int32 [E+1].
 * workspace: device, >= minite_workspace_bytes(MINITE_OP_QUANTIZE_TOKENS, E,
 *            row_src && !row_amax ? x_rows : 0), 4-byte aligned (per-expert
 *            maxima, and for gathered rows without row_amax one maximum per
 *            source row).
 * Device checks: offsets that do not start at 0, decrease or pass m_cap,
 * and kofs[E] > k_cap make the kernels write nothing; a row_src entry
 * outside [0, x_rows) reads as zeros; each sets bit 1<<MINITE_ERR_INVALID_ARG.
 * Shape rules: C % 16 == 0, 16 <= C <= 65536, 1 <= E <= 1024,
 * x_rows, m_cap < 2^31.
 */
int minite_quantize_tokens_nvfp4(const void* x, int64_t x_rows, const int32_t* row_src,
                                 const float* row_amax, int64_t m_cap, int64_t C, int32_t E,
                                 const int32_t* expert_offsets, int64_t k_cap, uint8_t* codes,
                                 uint8_t* sf, float* g_out, int32_t* kofs_out, void* workspace,
                                 size_t ws_bytes, int32_t* status, minite_stream_t stream);

/* Workspace bytes needed by `op` (MINITE_OP_QUANTIZE: a = groups;
 * MINITE_OP_PERMUTE_QUANT: a = T, b = H, E, k; MINITE_OP_COMBINE_BACKWARD_QUANT:
 * a = T, b = H; MINITE_OP_QUANTIZE_TOKENS: a = E, b = source rows when
 * they are gathered and no row maxima are passed, else 0;
 * MINITE_OP_GATE_UP_SWIGLU: a = M_total, b = I). 0 means none needed. */
size_t minite_workspace_bytes(int op, int64_t a, int64_t b, int32_t E, int32_t k);

/* Static description of a status code. */
const char* minite_status_string(int status);

/* Library version, "major.minor.patch". */
const char* minite_version(void);

/*
 * Test hooks: the element-wise converters and the specified exponential
 * exactly as the kernels above use them, over n values, so that they can be
 * compared with an independent CPU implementation across the whole float32
 * range. out_e2m1 receives one 4-bit code per byte; out_e4m3 one code per
 * byte (inputs must be >= 0 and finite).
 */
int minite_test_convert(const float* in, int64_t n, uint8_t* out_e2m1, uint8_t* out_e4m3,
                        float* out_exp, minite_stream_t stream);

/*
 * Test hook: digests of the element converters over every float32 bit
 * pattern, so that a test can compare them with a CPU reference on all 2^32
 * inputs without moving the results. Chunk c holds the patterns
 * [c * 2^20, (c + 1) * 2^20); for each chunk in [first_chunk, first_chunk +
 * n_chunks) this adds into digests[3 * (c - first_chunk) + j] (device,
 * caller zeroes) the sum modulo 2^64 of SplitMix64(((pattern << 32) |
 * result) ^ salt_j) over the chunk's finite inputs: j = 0 the E2M1 code
 * (salt 0x243F6A8885A308D3), j = 1 the E4M3 scale code of +0 and the
 * positive inputs (salt 0x13198A2E03707344), j = 2 the bits of the
 * specified exponential (salt 0xA4093822299F31D0). The converters are the
 * ones the kernels use. Returns MINITE_ERR_INVALID_ARG when the range
 * passes chunk 4095 or n_chunks exceeds 65536.
 */
int minite_test_convert_digest(unsigned long long first_chunk, unsigned long long n_chunks,
                               unsigned long long* digests, minite_stream_t stream);

/*
 * Test hook: the quantizers divide a block amax by 6 with an FMA-corrected
 * division by a constant instead of an IEEE division. This adds, into the
 * device counter *mismatches (caller zeroes it), the number of non-negative
 * finite floats x for which that result differs from the IEEE quotient x / 6
 * (expected: 0).
 */
int minite_test_div6_exhaustive(unsigned long long* mismatches, minite_stream_t stream);

/*
 * Test hook for failure detection: sets the time budget of every bounded
 * pipeline wait (the GEMM and the streaming kernels that stage rows through
 * shared memory with asynchronous copies; nanoseconds; 0 restores the
 * default of 2 s). A wait that runs out sets status bit 1<<MINITE_ERR_TIMEOUT
 * and the kernel returns after its in-flight copies have landed.
 * Process-wide; takes effect at the next launch.
 */
void minite_set_wait_budget_ns(uint64_t ns);

/*
 * Test hook: which grouped-GEMM kernel minite_grouped_gemm_nvfp4 launches.
 * 0 = automatic (currently 6 where it applies, else 1), 1 = single-CTA kernel
 * (128 x 256 tiles, one-chunk stages), 5 = single-CTA kernel with two-chunk
 * stages (K a multiple of 256 and at most about 830 experts; otherwise the
 * single-CTA kernel runs), 6 = CTA-pair kernel (256 x 256 tiles on the two
 * SMs of a cluster, five stages; at most about 1000 experts). Any other value
 * selects automatic. All give identical results.
 * Process-wide; takes effect at the next call.
 */
void minite_set_gemm_variant(int variant);

#ifdef __cplusplus
}
#endif

#endif /* MINITE_H */

/*
 * nf4.h -- C ABI of the GB300 (sm_103a) fused NF4 dequantise-and-multiply library.
 *
 * The operations are those of a frozen 4-bit Linear layer as the bitsandbytes
 * pages describe it:
 *   - quantize_4bit(w, blocksize=64, quant_type="nf4", compress_statistics=True)
 *     (bitsandbytes issue "MatMul4Bit keeps B and quant_state on ctx ...",
 *     section "Minimal reproducer");
 *   - dequantize_4bit(B, state), and the state's tensors absmax, offset, code,
 *     nested_absmax, nested_offset (same issue, sections "Root cause" and "Why
 *     save_for_backward fixes it");
 *   - the forward y = x W^T and the input gradient grad_x = grad_y W computed with
 *     no dense weight materialised (Soup issue #842, "Design sketch"; frozen base,
 *     "Scope"), with a deterministic reduction (same section: no atomics, no
 *     non-deterministic split-K);
 *   - a grouped per-expert variant (fork PR "Experts trainability ...", commits 1
 *     and 2).
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless a parameter says otherwise.  The caller
 *     owns every buffer (inputs, outputs and workspace); the library never
 *     allocates, frees or synchronises inside these calls.
 *   - `stream` is a cudaStream_t passed as void*; all work is enqueued on it,
 *     asynchronously.  NULL means the legacy default stream.
 *   - Arguments are validated on the host before anything is launched; a failed
 *     check returns an error status and launches nothing.  A CUDA launch failure
 *     returns NF4_ERR_CUDA.
 *   - Every device-side wait inside the kernels is bounded; a wait that runs out
 *     records NF4_ERR_TIMEOUT in a device status word (nf4_device_status) and the
 *     kernel returns instead of hanging.
 *   - Results are bit-identical from run to run for identical inputs, on a given
 *     device (the tile schedule depends only on the shapes and the SM count).
 *   - Weight layout: W is [N, K] row-major (out_features x in_features), flattened
 *     as i = n*K + k.  Blocks are consecutive runs of `blocksize` (64) values of
 *     the flat array; nested blocks are consecutive runs of `nested_blocksize`
 *     (256) blocks.  Packed byte j holds value 2j in its HIGH nibble and value 2j+1
 *     in its LOW nibble.
 *   - Activations and outputs are bf16, row-major with a leading dimension in
 *     elements.
 */
#ifndef NF4_GB300_H
#define NF4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NF4_OK = 0,
  NF4_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum value      */
  NF4_ERR_UNSUPPORTED_SHAPE = 2, /* e.g. K % 64 != 0 for the products                */
  NF4_ERR_ALIGNMENT = 3,         /* pointer or leading dimension not 16-byte aligned */
  NF4_ERR_WORKSPACE = 4,         /* workspace smaller than nf4_workspace_size()      */
  NF4_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed              */
  NF4_ERR_TIMEOUT = 6,           /* a bounded device wait ran out (device status)    */
  NF4_ERR_UNSUPPORTED = 7,       /* no sm_100-family device, or feature not built    */
  NF4_ERR_BAD_OFFSETS = 8,       /* grouped: expert offsets not monotone / in range  */
  NF4_ERR_BOUNDS = 9             /* checked build: an in-kernel index check failed   */
} nf4_status;

enum { NF4_DTYPE_F32 = 0, NF4_DTYPE_BF16 = 1 };

enum {
  NF4_OP_QUANTIZE = 0,
  NF4_OP_LINEAR_FWD = 1,
  NF4_OP_LINEAR_DGRAD = 2,
  NF4_OP_GROUPED_FWD = 3,
  NF4_OP_GROUPED_DGRAD = 4,
  NF4_OP_GROUPED_SWIGLU_BWD = 5  /* M = T rows, N = N_e, K; E experts */
};

/* Path counters (nf4_get_path_counters): how many launches each kernel got.
 * They prove which path produced a result (Soup issue #842, "Acceptance
 * criteria": report with a counter proving which path actually ran). */
enum {
  NF4_PATH_LINEAR_FWD = 0,   /* fused tcgen05 forward                      */
  NF4_PATH_LINEAR_DGRAD = 1, /* fused tcgen05 input gradient               */
  NF4_PATH_SPLITK_REDUCE = 2,/* fixed-order reduction of split partials    */
  NF4_PATH_GROUPED_FWD = 3,
  NF4_PATH_GROUPED_DGRAD = 4,
  NF4_PATH_DEQUANTIZE = 5,
  NF4_PATH_QUANTIZE = 6,
  NF4_PATH_TOTAL = 7,        /* every launch of the library                */
  NF4_PATH_GEMV_FWD = 8,     /* small-M SIMT forward                       */
  NF4_PATH_GEMV_DGRAD = 9,   /* small-M SIMT input gradient                */
  NF4_PATH_SKINNY_FWD = 10,  /* small-M tensor-core (mma.sync) forward     */
  NF4_PATH_SKINNY_DGRAD = 11,/* small-M tensor-core input gradient         */
  NF4_PATH_STREAM_K = 12,    /* fused launch with the stream-K schedule     */
  NF4_PATH_CLUSTER_SPLIT = 13,/* fused launch with the cluster split         */
  NF4_PATH_MULTI = 14,       /* multi-product fused launch                  */
  NF4_PATH_MOE_COMBINE = 15, /* top-k combine of the experts, or its backward */
  NF4_NUM_PATHS = 16
};

/* A quantised weight: the tensors of the pages' QuantState as plain device
 * pointers.  All are owned by the caller.
 *   packed         [ceil(N*K/2)] uint8, two 4-bit codes per byte (high = even).
 *   absmax         [nblocks] fp32 block absmax, nblocks = ceil(N*K/blocksize);
 *                  used when double_quant == 0 (may be NULL otherwise).
 *   absmax_q       [nblocks] uint8 8-bit codes of the absmax (double_quant == 1).
 *   nested_absmax  [ceil(nblocks/nested_blocksize)] fp32 (double_quant == 1).
 *   nested_offset  [1] fp32, the mean offset (double_quant == 1).
 *   code4          [16] fp32 4-bit codebook in ascending order with an exact zero:
 *                  the NF4 levels, or the E2M1 ("fp4") levels scaled to +-1 (whose
 *                  -0, +0 pair is the one repeated value).  Quantisation picks the
 *                  nearest level, ties to the lower index.
 *   code8          [256] fp32 8-bit map of the nested codes (double_quant == 1).
 * Decoded block scale under double quantisation (two roundings, no FMA):
 *   absmax'[b] = fp32(fp32(code8[absmax_q[b]] * nested_absmax[b/256]) + offset).
 * Dequantised value: fp32(code4[q] * absmax'[block]); the products use its bf16
 * rounding (round to nearest even) as the GEMM operand. */
typedef struct {
  const uint8_t* packed;
  const float* absmax;
  const uint8_t* absmax_q;
  const float* nested_absmax;
  const float* nested_offset;
  const float* code4;
  const float* code8;
  int64_t N;
  int64_t K;
  int32_t blocksize;        /* must be 64 */
  int32_t nested_blocksize; /* must be 256 when double_quant */
  int32_t double_quant;     /* 0 or 1 */
  int32_t bits;             /* code width: 4 (or 0, meaning 4) or 8.  With 8 the
                             * codes are one byte per value, packed [N*K], and
                             * code4 is the [256] value codebook (blockwise int8
                             * dynamic map or e4m3 levels) */
} nf4_weight;

/* nf4_quantize -- blockwise NF4 quantisation of W (quantize_4bit of bitsandbytes
 * issue "MatMul4Bit keeps B and quant_state on ctx", "Minimal reproducer"), with
 * optional double quantisation of the absmax (compress_statistics=True; "Root
 * cause").  Offline step, bit-exact with the CPU oracle.
 *   W        [numel = N*K] device array, fp32 or bf16 (w_dtype).
 *   blocksize 64.  Any numel >= 1; the last block may be short.
 *   Per block: a = max|w|; v = w / a (IEEE division); code = nearest level of
 *   code4 by fp64 midpoints, ties to the lower index; a == 0 -> index of the 0.
 *   Outputs: packed [ceil(numel/2)], absmax [nblocks] (always written), and when
 *   double_quant: absmax_q [nblocks], nested_absmax [ceil(nblocks/256)],
 *   nested_offset [1] (offset = fp32 of the mean of absmax, summed in fp64 over
 *   chunks of 1024 then over chunk sums; residuals quantised to code8 by nearest
 *   level, per nested block of 256 scaled by the residuals' max magnitude).
 *   ws: device workspace of nf4_workspace_size(NF4_OP_QUANTIZE, 0, N, K, 0) bytes
 *   (fp64 chunk sums; may be NULL when double_quant == 0). */
nf4_status nf4_quantize(const void* W, int32_t w_dtype, int64_t N, int64_t K, int32_t blocksize,
                        int32_t double_quant, int32_t nested_blocksize, const float* code4,
                        const float* code8, uint8_t* packed, float* absmax, uint8_t* absmax_q,
                        float* nested_absmax, float* nested_offset, void* ws, size_t ws_bytes,
                        void* stream);

/* nf4_quantize_8bit -- blockwise 8-bit storage of W, one code per byte (fork PR
 * "Experts trainability", commit 1, quant_type table: "int8: blockwise dynamic
 * map, 1 byte/value"; "fp8: e4m3 codebook, same blockwise path").  The same steps
 * and outputs as nf4_quantize with a 256-level codebook `code` (ascending, with
 * an exact zero; the e4m3 levels repeat only the signed zero) and codes [N*K]
 * instead of packed nibbles; double quantisation of the absmax as there.  The
 * products, dequantisation and grouped calls take the result as an nf4_weight
 * with bits = 8, packed = codes and code4 = code. */
nf4_status nf4_quantize_8bit(const void* W, int32_t w_dtype, int64_t N, int64_t K,
                             int32_t blocksize, int32_t double_quant, int32_t nested_blocksize,
                             const float* code, const float* code8, uint8_t* codes,
                             float* absmax, uint8_t* absmax_q, float* nested_absmax,
                             float* nested_offset, void* ws, size_t ws_bytes, void* stream);

/* nf4_dequantize -- dense dequantisation of a quantised weight (dequantize_4bit,
 * bitsandbytes issue "MatMul4Bit keeps B and quant_state on ctx", "Root cause").
 * Not on the fused path; provided for checks and for callers that need a dense
 * copy.  out: [N*K] fp32 (value wf) or bf16 (round-to-nearest-even of wf),
 * per out_dtype.  Bit-exact with the oracle. */
nf4_status nf4_dequantize(const nf4_weight* w, void* out, int32_t out_dtype, void* stream);

/* nf4_linear_fwd -- fused forward y = x W^T straight from the packed codes and the
 * (nested) statistics; the dequantised bf16 tile exists only in shared memory
 * (Soup issue #842, "Design sketch").
 *   x  [M, K] bf16, leading dimension ldx (elements, multiple of 8, ldx >= K).
 *   y  [M, N] bf16, leading dimension ldy (>= N).
 *   M >= 0 (M == 0 is a no-op); K % 64 == 0; x 16-byte aligned.
 *   ws: device workspace of nf4_workspace_size(NF4_OP_LINEAR_FWD, M, N, K, 0)
 *   bytes (split-K partials for small M; may be NULL when that size is 0).
 *   Paths (nf4_get_path_counters tells which ran): M <= 16 runs the warp-MMA
 *   small-M kernels for 4-bit codes (mma.sync, fixed-order cluster reduction; see
 *   nf4_set_small_m_path for the SIMT GEMV and tiled alternatives); larger M, and
 *   every M for 8-bit codes, runs the tcgen05 kernel (fp32
 *   accumulation in tensor memory) with the classic or stream-K schedule
 *   (nf4_set_stream_k).  Split partials are summed in a fixed order, by a second
 *   kernel (classic) or by the CTA finishing the tile (stream-K).  No atomics. */
nf4_status nf4_linear_fwd(const void* x, int64_t M, int64_t ldx, const nf4_weight* w, void* y,
                          int64_t ldy, void* ws, size_t ws_bytes, void* stream);

/* nf4_linear_dgrad -- fused input gradient grad_x = grad_y W (the backward of
 * MatMul4Bit, bitsandbytes issue "MatMul4Bit keeps B and quant_state on ctx",
 * "Root cause"; only grad_x since the base is frozen, Soup issue #842 "Scope").
 *   gy [M, N] bf16, leading dimension ldgy (multiple of 8, >= N).
 *   gx [M, K] bf16, leading dimension ldgx (>= K).
 *   Same rules as nf4_linear_fwd (the SIMT path serves M <= 4); workspace from
 *   NF4_OP_LINEAR_DGRAD. */
nf4_status nf4_linear_dgrad(const void* gy, int64_t M, int64_t ldgy, const nf4_weight* w, void* gx,
                            int64_t ldgx, void* ws, size_t ws_bytes, void* stream);

/* nf4_linear_fwd_multi / nf4_linear_dgrad_multi -- up to NF4_MAX_MULTI
 * independent products of nf4_linear_fwd / nf4_linear_dgrad in ONE launch of the
 * fused tcgen05 kernel, for products that become ready together (for instance
 * the q, k and v projections of one input, or gate and up): product p computes
 *   forward:        y[p]  = x[p] W[p]^T   (x[p] [M, K], y[p] [M, N_p]),
 *   input gradient: gx[p] = gy[p] W[p]    (gy[p] [M, N_p], gx[p] [M, K]),
 * each exactly as the single-product call computes it (same operands, fp32
 * accumulation in tensor memory, bf16 output, bit-identical reruns), but the
 * products' work items share one grid, so a small product no longer pays a whole
 * launch's start-up and drain.  The arrays are host arrays of nprod entries
 * (device pointers, leading dimensions in elements); the x pointers may be equal.
 * Requirements: 1 <= nprod <= NF4_MAX_MULTI; the same M and K for every product;
 * 4-bit codes, the same double_quant setting and the same code4 / code8 tables
 * (pointer-equal) for every weight; bf16 activations and outputs; K % 64 == 0;
 * activations, outputs and packed codes 16-byte aligned with leading dimensions
 * multiples of 8 (NF4_ERR_ALIGNMENT otherwise); no workspace.  M == 0 is a
 * no-op.  Products are scheduled in order of decreasing contraction length with
 * the classic schedule and 128- or 256-token tiles (a deterministic function of
 * the shapes and the SM count). */
#define NF4_MAX_MULTI 4
nf4_status nf4_linear_fwd_multi(int32_t nprod, const void* const* x, int64_t M, const int64_t* ldx,
                                const nf4_weight* const* w, void* const* y, const int64_t* ldy,
                                void* stream);
nf4_status nf4_linear_dgrad_multi(int32_t nprod, const void* const* gy, int64_t M, const int64_t* ldgy,
                                  const nf4_weight* const* w, void* const* gx, const int64_t* ldgx,
                                  void* stream);

/* nf4_moe_combine -- the top-k combine of the grouped experts: the grouped
 * products leave one bf16 row per (token, routed expert), rows [R, H] (row pitch
 * ld_rows), typically after the down projection with the routing weights applied
 * as its row scale (nf4_grouped_fwd_ep); token t's output is the sum of its rows
 *   out[t][c] = bf16( sum_{j < k, token_rows[t*k + j] >= 0} rows[token_rows[t*k + j]][c] )
 * in fp32, in route order j, rounded once (round to nearest even); deterministic.
 * token_rows: device int32 [tokens, k], the row of each (token, route), -1 for an
 * absent route; an index >= R is skipped and recorded as NF4_ERR_BAD_OFFSETS in
 * the device status word.  out [tokens, H] bf16 (row pitch ld_out).  H % 8 == 0,
 * rows / out 16-byte aligned with pitches multiples of 8 (NF4_ERR_ALIGNMENT),
 * k >= 1, tokens, R >= 0 (tokens == 0 or H == 0: nothing to do).
 * nf4_moe_combine_bwd -- its backward: grad_rows[token_rows[t*k + j]] =
 * grad_out[t] (an exact copy) for every present route; rows that no route names
 * are not written.  grad_out [tokens, H] (pitch ld_grad_out), grad_rows [R, H]
 * (pitch ld_grad_rows); the same requirements. */
nf4_status nf4_moe_combine(const void* rows, int64_t R, int64_t ld_rows, const int32_t* token_rows,
                           int64_t tokens, int32_t k, int64_t H, void* out, int64_t ld_out, void* stream);
nf4_status nf4_moe_combine_bwd(const void* grad_out, int64_t tokens, int64_t ld_grad_out,
                               const int32_t* token_rows, int32_t k, int64_t R, int64_t H, void* grad_rows,
                               int64_t ld_grad_rows, void* stream);

/* nf4_linear_fwd_f16 / nf4_linear_dgrad_f16 -- the same products for the fp16
 * compute dtype (Soup issue #842, "Design sketch": keep the dtype handling of
 * Linear4bit, which computes in the activations' half-precision type): x / grad_y
 * and y / grad_x are IEEE fp16, and the operand is fp16(fp32(code4[q] * absmax'))
 * (round to nearest even) instead of bf16.  Same arguments, workspace and
 * determinism as nf4_linear_fwd / nf4_linear_dgrad; M <= 16 runs the warp-MMA
 * small-M kernels with fp16 MMAs (the SIMT GEMV alternative is bf16 only, so
 * NF4_SMALL_M_SIMT sends fp16 to the fused kernel), larger M the fused tcgen05
 * kernel (fp16 tcgen05 MMAs); fp32 accumulation throughout.  4-bit codes only
 * (bits == 8 -> NF4_ERR_UNSUPPORTED). */
nf4_status nf4_linear_fwd_f16(const void* x, int64_t M, int64_t ldx, const nf4_weight* w, void* y,
                              int64_t ldy, void* ws, size_t ws_bytes, void* stream);
nf4_status nf4_linear_dgrad_f16(const void* gy, int64_t M, int64_t ldgy, const nf4_weight* w,
                                void* gx, int64_t ldgx, void* ws, size_t ws_bytes, void* stream);

/* nf4_grouped_fwd -- per-expert forward for a stack of E frozen experts quantised
 * as one tensor (fork PR "Experts trainability ...", commit 1: the fused 3-D
 * expert stack; commit 2: no dequantised weight is kept).
 *   w        the stacked weight: w->N == E * N_e rows, expert e owns rows
 *            [e*N_e, (e+1)*N_e); w->K = K.
 *   offsets  DEVICE int32 [E+1]: rows offsets[e] .. offsets[e+1]-1 of x belong to
 *            expert e; offsets[0] == 0, non-decreasing, offsets[E] == T.  Offsets
 *            outside that contract are detected on the device: the bad expert's
 *            rows are skipped and NF4_ERR_BAD_OFFSETS is recorded in the device
 *            status word.
 *   x [T, K] bf16 (ldx), y [T, N_e] bf16 (ldy).  No workspace is needed. */
nf4_status nf4_grouped_fwd(const void* x, const int32_t* offsets, int32_t E, int64_t T, int64_t ldx,
                           const nf4_weight* w, int64_t N_e, void* y, int64_t ldy, void* stream);

/* nf4_grouped_fwd_ep -- nf4_grouped_fwd with the expert epilogue fused into the
 * kernel (fork PR "Experts trainability" and Soup issue #842 run these in torch
 * around the products): with a = x_e W_e^T per expert,
 *   bias       [E*N_e] fp32 added per weight row (NULL: none);
 *   swiglu     1: the weight rows of each expert are interleaved in groups of 128,
 *              64 gate rows then the 64 up rows of the same output columns (N_e a
 *              multiple of 128); y has N_e/2 columns, y = silu(g) * u with
 *              silu(g) = g / (1 + exp(-g)), g and u including their biases;
 *              0: y = a (+ bias), N_e columns;
 *   row_scale  [T] fp32 multiplying each output row last (the tokens' routing
 *              weights in the expert-sorted order; NULL: none).
 * fp32 arithmetic, one bf16 rounding at the end; otherwise as nf4_grouped_fwd. */
typedef struct {
  const float* bias;
  const float* row_scale;
  int32_t swiglu;
} nf4_epilogue;
nf4_status nf4_grouped_fwd_ep(const void* x, const int32_t* offsets, int32_t E, int64_t T,
                              int64_t ldx, const nf4_weight* w, int64_t N_e, const nf4_epilogue* ep,
                              void* y, int64_t ldy, void* stream);

/* nf4_grouped_dgrad -- per-expert input gradient gx[rows of e] = gy[rows of e] W_e.
 *   gy [T, N_e] bf16 (ldgy), gx [T, K] bf16 (ldgx); other arguments as above. */
nf4_status nf4_grouped_dgrad(const void* gy, const int32_t* offsets, int32_t E, int64_t T,
                             int64_t ldgy, const nf4_weight* w, int64_t N_e, void* gx, int64_t ldgx,
                             void* stream);

/* nf4_grouped_swiglu_bwd -- backward of nf4_grouped_fwd_ep with swiglu = 1 (fork
 * PR "Experts trainability ...", commit 2: the backward recomputes the expert
 * products from the frozen 4-bit weight and keeps no dequantised weight).  With
 * h = silu(g) * u * r (r = row_scale[t], or 1), given the upstream gradient gh:
 *   1. the grouped forward product is recomputed over the interleaved gate/up
 *      weight and its epilogue forms, in fp32, s = 1 / (1 + exp(-g)),
 *      dg = gh r u s (1 + g (1 - s)) and du = gh r g s, rounded to bf16 into the
 *      workspace at the gate and up rows' own columns ([T, N_e]);
 *   2. one grouped input-gradient product over the same weight turns them into
 *      gx = [dg du]_e W_e for each expert's rows;
 *   3. with grad_row_scale (needs ep->row_scale): grad_row_scale[t] = sum over
 *      the row's N_e/2 outputs of silu(g) u gh, as fp32 partials per 32 gate
 *      columns added in a fixed order (rows outside the expert ranges get 0).
 *   x [T, K] bf16 (ldx), the forward's input; w, offsets, E, N_e, ep (swiglu must
 *   be 1; bias and row_scale as in the forward) as in nf4_grouped_fwd_ep.
 *   gh [T, N_e/2] bf16 (ldgh, a multiple of 8, 16-byte aligned); gx [T, K] bf16
 *   (ldgx); grad_row_scale DEVICE fp32 [T] or NULL.
 *   ws: device workspace of nf4_workspace_size(NF4_OP_GROUPED_SWIGLU_BWD, T, N_e,
 *   K, E) bytes, 256-byte aligned (NF4_ERR_WORKSPACE / NF4_ERR_ALIGNMENT).
 * Deterministic: no atomics; every output has a fixed summation order.  Returns
 * NF4_ERR_INVALID_ARG for swiglu != 1, grad_row_scale without row_scale, or the
 * argument errors of the grouped products. */
nf4_status nf4_grouped_swiglu_bwd(const void* x, const int32_t* offsets, int32_t E, int64_t T,
                                  int64_t ldx, const nf4_weight* w, int64_t N_e,
                                  const nf4_epilogue* ep, const void* gh, int64_t ldgh, void* gx,
                                  int64_t ldgx, float* grad_row_scale, void* ws, size_t ws_bytes,
                                  void* stream);

/* nf4_linear_fwd_noalloc -- the forward of nf4_linear_fwd without a workspace
 * argument, for callers that cannot allocate device memory themselves (for
 * instance code running under a framework allocator that owns all device memory,
 * or a plugin that is handed only its input and output buffers).  The pages
 * have no counterpart: it is a deployment variant of the same computation.
 *   Arguments, layouts and results are those of nf4_linear_fwd (same kernels,
 *   same tile plan, same outputs).
 *   Scratch: the split-contraction partials go to a fixed file-scope device
 *   array of NF4_NOALLOC_SCRATCH_BYTES (2 MiB), which every GPU that loads the
 *   library holds until the process exits.  Shapes whose partials need more
 *   return NF4_ERR_WORKSPACE and launch nothing; the call never allocates.
 *   Set-up: the first call on a device looks up the array's device address
 *   (with that device current); make that first call before any stream capture.
 *   Sharing: all calls use the same array and it keeps the last call's
 *   contents; a call writes every partial before reading it, so nothing needs
 *   clearing.  Calls that overlap on the GPU (for instance on two streams of
 *   one device) race on that device's array: serialise them.  Each device holds
 *   its own copy. */
#define NF4_NOALLOC_SCRATCH_BYTES (2u << 20)
nf4_status nf4_linear_fwd_noalloc(const void* x, int64_t M, int64_t ldx, const nf4_weight* w,
                                  void* y, int64_t ldy, void* stream);

/* Workspace bytes an operation needs for the given shape on the current device
 * (0 when none).  op is one of NF4_OP_*; E is unused for the dense products. */
size_t nf4_workspace_size(int32_t op, int64_t M, int64_t N, int64_t K, int32_t E);

/* Static string naming a status code. */
const char* nf4_status_string(nf4_status s);

/* 1 when this library is the checked debug build (libnf4_checked.so, compiled
 * with NF4_CHECKED=1), else 0.  The checked build tests the indices of the
 * kernels' computed global and shared-memory accesses (statistics loads, the
 * output, split and stream-K partial stores, the small-M kernels' loads and
 * stores, the decoders' shared-memory offsets) before each access; an index
 * outside its buffer skips that access and records NF4_ERR_BOUNDS in the device
 * status word (nf4_device_status).  It stands in for a memory checker on devices
 * where none can run; results are otherwise those of the normal build. */
int32_t nf4_checked_build(void);

/* Copies the NF4_NUM_PATHS host-side launch counters into out (host array of
 * NF4_NUM_PATHS entries). */
void nf4_get_path_counters(uint64_t* out);
void nf4_reset_path_counters(void);

/* Reads (and with clear != 0, resets) the device status word of the current
 * device into *out (host int).  Synchronises with the device; not for hot paths. */
nf4_status nf4_device_status(int32_t* out, int32_t clear);

/* Declares (enabled != 0) that no kernel running just before a product call on
 * the same stream writes that call's weight tensors (packed codes, statistics,
 * codebooks), as holds for a frozen weight.  The product kernels are launched
 * with programmatic dependent launch: they start while the previous kernel on
 * the stream drains and wait for it before they read activations or write
 * outputs.  With this declaration the small-M kernels and the dense fused
 * kernel also read the weight before that wait (the fused kernel's code stream
 * and decode of its first steps then overlap the previous kernel's tail; the
 * grouped products keep every read after the wait).  Off by default (every read
 * then follows the wait).  Results do not depend on the setting. */
void nf4_set_weight_prefetch(int32_t enabled);

/* Kernels for the dense products at small M (M <= 16), for comparisons and tests:
 *   NF4_SMALL_M_AUTO  (default) the tensor-core small-M kernels (warp-level bf16
 *                     MMA over a shared dequantisation table, contraction split
 *                     across thread-block clusters) where their plan fits, else
 *                     as below;
 *   NF4_SMALL_M_SIMT  the SIMT GEMV kernels for M <= 4, the tiled tcgen05
 *                     kernels above;
 *   NF4_SMALL_M_TILES the tiled tcgen05 kernels with a split contraction.
 * Every choice is deterministic; results may differ in the last bit between
 * choices (different fp32 summation grouping). */
enum { NF4_SMALL_M_AUTO = 0, NF4_SMALL_M_SIMT = 1, NF4_SMALL_M_TILES = 2 };
void nf4_set_small_m_path(int32_t path);

/* Schedule of the fused tcgen05 kernel for the dense products (process-wide;
 * host only).  Classic: every CTA takes whole tiles (with a fixed contraction
 * split at small M), leaving the last wave partly idle when the tile count is not
 * a multiple of the SM count.  Stream-K: the tiles' 64-deep contraction steps are
 * cut into one equal contiguous run per CTA; a tile cut between CTAs is finished
 * by the highest-index CTA holding part of it, which adds the lower CTAs' fp32
 * partial tiles in a fixed order (deterministic for a given shape and SM count).
 * The workspace then holds the partials (CTAs x 128 x tile-tokens fp32) and one
 * 8-byte ready flag per CTA and row quarter; concurrent calls need workspaces of
 * their own, as for the split partials.
 *   NF4_STREAM_K_OFF   classic only.
 *   NF4_STREAM_K_AUTO  (default) stream-K where the planner's cost model prefers it.
 *   NF4_STREAM_K_FORCE stream-K for every product on the fused kernel (tests).
 * A CTA waits (bounded, NF4_ERR_TIMEOUT on expiry) only for partials of CTAs of
 * lower index, which the device dispatches before it, so the grid need not be
 * resident at once: other kernels may share the device (for instance a second
 * stream-K product on another stream). */
enum { NF4_STREAM_K_OFF = 0, NF4_STREAM_K_AUTO = 1, NF4_STREAM_K_FORCE = 2 };
void nf4_set_stream_k(int32_t mode);

/* Cluster split of the fused tcgen05 kernel for the dense products (process-wide;
 * host only): when every tile of a product, cut into S contraction slices (S = 2,
 * 4 or 8, at least 32 tokens of the tile per slice), fits the device in one wave
 * of thread-block clusters of S CTAs, the S slices of a tile run on the CTAs of
 * one cluster.  Cluster rank p then finishes token slice p of the tile: every rank
 * writes its fp32 partial of the other slices into their owners' shared memory
 * (distributed shared memory), and the owner adds the S partials in rank order
 * and stores bf16.  No workspace, no partials in global memory, no reduction
 * kernel; deterministic for a given shape and device.  Needs a 16-byte aligned
 * output and row pitch; 4-bit codes.
 *   NF4_CLUSTER_SPLIT_OFF   never.
 *   NF4_CLUSTER_SPLIT_AUTO  (default) where the planner's cost model prefers it.
 *   NF4_CLUSTER_SPLIT_FORCE wherever it applies (tests). */
enum { NF4_CLUSTER_SPLIT_OFF = 0, NF4_CLUSTER_SPLIT_AUTO = 1, NF4_CLUSTER_SPLIT_FORCE = 2 };
void nf4_set_cluster_split(int32_t mode);

/* Token tile of the fused tcgen05 kernel for the dense products (process-wide;
 * host only): 0 (default) lets the planner choose; 64, 128, 256 or 512 fixes it
 * for every product with M > 32 that runs on the fused kernel (8-bit codes: at
 * most 128).  512 is the CTA-pair tile: the two CTAs of a thread-block cluster
 * share each 256-row MMA (cta_group::2), each decoding its 128 weight rows and
 * holding 128 tokens of each 256-token half, two MMAs per contraction step into
 * a 512-column accumulator per CTA (classic schedule only; the planner takes it
 * from M = 1024 where its cost model prefers it).  For tests and measurements.
 * Other values are ignored. */
void nf4_set_token_tile(int32_t tokens);

/* The launch plan a dense product (NF4_OP_LINEAR_FWD / NF4_OP_LINEAR_DGRAD)
 * takes, computed on the host without a device: a deterministic function of the
 * shape, the SM count `sms`, the code width `bits` (4 or 8), the compute dtype
 * (`f16` != 0: fp16) and the process-wide launch options (nf4_set_stream_k,
 * nf4_set_small_m_path, nf4_set_cluster_split, nf4_set_token_tile).  With a current device the
 * cluster split also takes the device's cluster residency into account.  For diagnostics and tests; the
 * product calls compute the same plan with the current device's SM count.
 * Returns NF4_ERR_INVALID_ARG for a null `out`, an unknown op, sms < 1,
 * bits other than 4 / 8, fp16 with 8-bit codes or a non-positive dimension. */
enum { NF4_PLAN_FUSED = 0, NF4_PLAN_SMALL_M_MMA = 1, NF4_PLAN_SIMT_GEMV = 2 };
typedef struct nf4_plan_info {
  int32_t kernel;          /* NF4_PLAN_*: tcgen05 tiles, warp-MMA small-M, SIMT GEMV   */
  int32_t token_tile;      /* fused: tokens per tile (16 .. 256; 512: CTA-pair tile)    */
  int32_t splits;          /* fused classic: contraction splits (1 = none)              */
  int32_t stream_k;        /* fused: 1 for the stream-K schedule                        */
  int32_t grid;            /* fused: CTAs launched; small-M MMA: clusters x CTAs per    */
                           /* cluster; 0 for the GEMV kernels (sized at launch)         */
  int64_t items;           /* fused: work items (tiles x splits)                        */
  uint64_t workspace_bytes;/* workspace this plan needs                                */
  int32_t cluster_split;   /* fused: CTAs of a cluster sharing each tile (splits), or 0 */
  int32_t tail_tokens;     /* fused token split: the last tail_tokens tokens run as a   */
                           /* second launch (the fields above describe the first        */
                           /* M - tail_tokens), or 0                                    */
  int32_t tail_token_tile; /* tokens per tile of that second launch (256), or 0          */
} nf4_plan_info;
nf4_status nf4_plan_query(int32_t op, int64_t M, int64_t N, int64_t K, int32_t sms, int32_t bits,
                          int32_t f16, nf4_plan_info* out);

/* Failure-path test hook (host-side injection; no fault of any kind): arms a
 * one-shot for the next stream-K launch of this process, whose finishing CTAs
 * then wait for a flag value that no CTA publishes.  Their bounded waits run out
 * (2 s), the kernel records NF4_ERR_TIMEOUT in the device status word
 * (nf4_device_status), finishes its remaining work with whatever the partials
 * hold, and exits normally; the device stays usable and later launches are
 * unaffected.  The affected call's output is unspecified. */
void nf4_inject_stream_k_timeout(void);

/* Failure-path test hook of the checked build (nf4_checked_build): one-shot for
 * the next product launched on the fused tcgen05 kernel (nf4_linear_* at an M
 * that takes it) by this process, whose statistics-load index checks then fail.
 * Each such load is skipped (its block reads as scale 0; nothing is accessed out
 * of range) and NF4_ERR_BOUNDS is recorded in the device status word; the kernel
 * finishes normally and later launches are unaffected.  The affected call's
 * output is unspecified.  No effect in the normal build. */
void nf4_inject_bounds_failure(void);

/* Human-readable message of the last CUDA error that made a call of this thread
 * return NF4_ERR_CUDA ("no error" if none).  Static string. */
const char* nf4_last_cuda_error(void);

/* Library and device information: returns NF4_OK when the current device is an
 * sm_100-family GPU the kernels were built for; *sm_count receives its SM count. */
nf4_status nf4_device_check(int32_t* sm_count);

#ifdef __cplusplus
}
#endif

#endif /* NF4_GB300_H */

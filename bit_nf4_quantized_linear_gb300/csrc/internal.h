// internal.h -- declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "nf4.h"

namespace nf4 {

// Device status codes written by kernels into the status word (same values as
// nf4_status).
constexpr int kStatusTimeout = NF4_ERR_TIMEOUT;
constexpr int kStatusBadOffsets = NF4_ERR_BAD_OFFSETS;

// Checked debug build (-DNF4_CHECKED=1, libnf4_checked.so): the kernels test the
// index of each computed global or shared-memory access with in_bounds() before
// it; a false test records NF4_ERR_BOUNDS in the status word (first error wins)
// and the caller skips the access.  In the normal build in_bounds() is the
// constant true and the tests compile to nothing.
#ifndef NF4_CHECKED
#define NF4_CHECKED 0
#endif

#ifdef __CUDACC__
__device__ __forceinline__ bool in_bounds(bool ok, int* status) {
#if NF4_CHECKED
  if (!ok && status) atomicCAS(status, 0, NF4_ERR_BOUNDS);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}
#endif

// Upper bound of experts the grouped kernels accept.
constexpr int kMaxExperts = 512;

// Tile geometry of the fused products.
constexpr int kTileW = 128;  // rows of the dequantised operand per tile (MMA M)
constexpr int kTileK = 64;   // contraction per pipeline stage (one 64-value block)

// Top-k combine of the grouped experts and its backward (nf4_moe_combine,
// nf4_moe_combine_bwd).  Forward: rows = the grouped output [R, H], out = [tokens,
// H]; backward: rows = the gradient of the combined output [tokens, H], out = the
// rows' gradient [R, H].  token_rows [tokens, k]: row of each (token, route), -1
// for none.
struct MoeArgs {
  const __nv_bfloat16* rows;
  int64_t ld_rows;
  const int32_t* token_rows;
  int32_t k;
  int64_t tokens, R, H;
  __nv_bfloat16* out;
  int64_t ld_out;
  int* status;
};
cudaError_t launch_moe(bool backward, const MoeArgs& a, cudaStream_t s);

// Multi-product launches (nf4_linear_fwd_multi / nf4_linear_dgrad_multi): up to
// kMaxProds independent products with the same M and in-features K, each with its
// own weight, activation and output, whose work items share one grid.
constexpr int kMaxProds = 4;

// One product of a multi-product launch.
struct ProdArgs {
  const float* absmax;
  const uint8_t* absmax_q;
  const float* nested_absmax;
  const float* nested_offset;
  __nv_bfloat16* out;
  int64_t ld_out;
  int64_t N_total;  // rows of this weight
  int64_t ncols;    // output columns (forward: this weight's rows; input gradient: K)
  int ksteps;       // contraction steps of an item
  int wtiles;       // tiles over the output columns
  int64_t item0;    // first item of this product in the launch's item order
};

// Tensor maps of a launch: activations, packed codes and output, one per product
// (N = 1 for single-product launches).
template <int N>
struct MapSet {
  CUtensorMap act[N];
  CUtensorMap pk[N];
  CUtensorMap out[N];
};

// Parameters of the fused product kernel (everything but the tensor maps).
struct GemmArgs {
  int64_t M;        // activation rows (dense) or T (grouped)
  int64_t ncols;    // output columns: N (fwd), N_e (grouped fwd), K (dgrad)
  int64_t N_total;  // rows of the packed weight tensor
  int64_t K;        // in-features
  int64_t KB;       // K / 64
  int64_t N_e;      // rows per expert (grouped); N for dense
  int ksteps;       // contraction steps of a full item
  int wtiles;       // tiles over the output columns
  int ttiles;       // token tiles (dense)
  int splits;       // contraction splits (dense, small M)
  int64_t total_items;  // dense only; grouped computes it on the device
  int grouped;
  int E;
  const int32_t* offsets;
  const float* absmax;
  const uint8_t* absmax_q;
  const float* nested_absmax;
  const float* nested_offset;
  const float* code4;
  const float* code8;
  int dq;
  __nv_bfloat16* out;
  int64_t ld_out;
  float* ws;  // split-K partials [splits][M][ncols]
  int* status;
  int prefetch;  // dense: the weight may be read before the preceding grid has finished
  int tma_out;  // dense bf16 output written by bulk tensor stores (aligned out and ld_out)
  // Cluster split (dense, tma_out): cs > 1 CTAs, one cluster, share each tile, one
  // contraction slice each (items = tiles x cs, one per CTA, splits == cs); token
  // slice p of the tile (bt / cs tokens) is summed and stored by cluster rank p from
  // the partials the other ranks write into its activation ring.
  int cs;
  // Grouped forward epilogue (nf4_grouped_fwd_ep): fp32 bias per weight row, fp32
  // scale per output row (routing weights), SwiGLU of interleaved gate/up rows.
  const float* ep_bias;
  const float* ep_scale;
  int ep_swiglu;
  // Backward of the SwiGLU epilogue (ep_swiglu and ep_bwd set): the recomputed
  // gate g and up u meet the upstream gradient dh [T, N_e / 2] (bf16, row pitch
  // ep_ld_dh) and, instead of h, the kernel writes dg = dh r u silu'(g) and
  // du = dh r silu(g) in bf16 at the weight rows' own columns of `out` ([T, N_e]),
  // and, when ep_drw is set, per 32 gate columns the fp32 partial sum over those
  // columns of silu(g) u dh into ep_drw[(N_e / 64) partials][T].
  int ep_bwd;
  const __nv_bfloat16* ep_dh;
  int64_t ep_ld_dh;
  float* ep_drw;
  // Stream-K schedule (dense, splits == 1): the items * ksteps
  // contraction steps are cut into sk_ctas equal contiguous runs, one per CTA, and
  // each CTA walks the tiles of its run in reverse.  A tile cut between CTAs is
  // finished by the highest-index CTA holding part of it (the one with its last
  // steps), which adds the lower CTAs' fp32 partials in a fixed order; a CTA thus
  // only ever waits for CTAs of lower index, which are dispatched before it.
  int sk;
  int64_t sk_units;     // items * ksteps
  int sk_ctas;          // CTAs (= grid)
  float* sk_ws;         // partial tiles [sk_ctas][4 row quarters][bt tokens][32 rows] fp32
  uint64_t* sk_flags;   // [sk_ctas][4] in the caller's workspace: partial of (CTA,
                        // row quarter) published; cleared by the finishing CTA
  uint64_t sk_epoch;    // value this launch publishes (never 0)
  uint64_t sk_wait_xor; // the finishing CTA waits for sk_epoch ^ sk_wait_xor (0; the
                        // failure-path test sets a bit no contributor publishes)
  int chk_inject;       // checked build: fail the statistics-load index check (test hook)
  // Multi-product launches: nprod products (items of product p from prod[p].item0),
  // classic schedule, no splits; the single-product fields above are unused for
  // the per-product quantities.
  int nprod;
  ProdArgs prod[kMaxProds];
};

// Stream-K workspace: partial tiles, then the ready flags (8 bytes per CTA and row
// quarter).
constexpr int kSkMaxCtas = 1024;
inline size_t stream_k_ws_bytes(int ctas, int bt) {
  return static_cast<size_t>(ctas) * kTileW * bt * sizeof(float) + static_cast<size_t>(ctas) * 4 * 8;
}

// Parameters of the small-M GEMV kernels.
struct GemvArgs {
  const __nv_bfloat16* act;  // x [M, K] (forward) or grad_y [M, N] (input gradient)
  int64_t ld_act;
  const uint8_t* packed;
  int64_t N, K, KB;
  const float* absmax;
  const uint8_t* absmax_q;
  const float* nested_absmax;
  const float* nested_offset;
  const float* code4;
  const float* code8;
  int dq;
  __nv_bfloat16* out;
  int64_t ld_out;
  float* ws;  // input gradient: per-row-group partials [groups][M][K]
  int64_t M;
  int64_t m0;  // first activation row of a launch (set by the launcher)
  int kseg;    // forward: contraction segments per row group
  int* status;
};

// Parameters of the small-M tensor-core kernels (mma.sync m16n8k16).  The grid
// is C clusters of S CTAs; cluster c owns the output tiles c*T/C .. (c+1)*T/C - 1
// (forward: 16 weight rows; input gradient: 64 in-features), and CTA rank r of a
// cluster owns the contraction slice r*cc .. (r+1)*cc - 1; the S partial sums of
// a tile are reduced through distributed shared memory in rank order.
// Shared-memory layout of a small-M CTA (byte offsets).
struct SkinnyLayout {
  int table, ring, gy, first, recv, scales, code8, bars, act, total;
};

struct SkinnyArgs {
  // x [M, K] (forward) or grad_y [M, N] (input gradient); like `out`, bf16, or
  // IEEE fp16 bits when f16 is set.
  const __nv_bfloat16* act;
  int64_t ld_act;
  const uint8_t* packed;
  int64_t N, K, KB;
  const float* absmax;
  const uint8_t* absmax_q;
  const float* nested_absmax;
  const float* nested_offset;
  const float* code4;
  const float* code8;
  int dq;
  int f16;        // fp16 operands and output
  __nv_bfloat16* out;
  int64_t ld_out;
  int64_t M;
  int S;          // CTAs per cluster (contraction split)
  int C;          // clusters
  int64_t T;      // output tiles
  int64_t cc;     // contraction per CTA (forward: multiple of 64; input gradient: of 16)
  int prefetch;   // the weight may be read before the preceding grid has finished
  int* status;    // device status word (NF4_ERR_TIMEOUT from a bounded wait)
  // Derived on the host by launch_skinny (no 64-bit divisions in the kernels):
  SkinnyLayout lay;  // the CTA's shared-memory layout
  int64_t nt_max;    // most tiles of a cluster, ceil(T / C)
  int64_t tq;        // T / C
  int tr;            // T % C
  int log2S;         // S = 1 << log2S
};

constexpr int kSkinnyMaxM = 16;

struct SkinnyPlan {
  int S = 0, C = 0;
  int64_t T = 0, cc = 0;
  size_t smem = 0;
};

// Plans and launches (S CTAs per cluster along the contraction).
bool skinny_plan(int mode, int64_t M, int64_t N, int64_t K, int sms, SkinnyPlan* p, bool f16 = false);
// tmap: the packed codes [N rows, K/2 bytes] as a uint8 tensor with a box of
// 128 bytes x 16 rows and 128B swizzle (forward) or 32 bytes x 64 rows and 32B
// swizzle (input gradient).
cudaError_t launch_skinny(int mode, const SkinnyArgs& a, const SkinnyPlan& p, const CUtensorMap& tmap,
                          cudaStream_t s);

// Largest M each product sends to the GEMV kernels.
constexpr int kGemvMaxMFwd = 4;
constexpr int kGemvMaxMDgrad = 4;

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_gemv_fwd(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_dgrad(const GemvArgs& a, cudaStream_t s);
int gemv_fwd_kseg(int64_t K);
int64_t gemv_dgrad_row_groups(int64_t N);
// tmap_out: 16-bit output [M, ncols] with a 32 x 32 box, used when a.tma_out is set.
// bits: code width of the weight (4, or 8 with bt <= 128).  f16: fp16 activations,
// operand and output instead of bf16 (4-bit codes).
// Multi-product launch (a.nprod products, bf16, 4-bit codes, bt 128 or 256,
// classic schedule); maps.act/pk/out[p] are product p's tensor maps.
cudaError_t launch_gemm_multi(int mode, int bt, const GemmArgs& a, const MapSet<kMaxProds>& maps, int grid,
                              cudaStream_t s);
cudaError_t launch_gemm(int mode, int bt, int bits, bool f16, const GemmArgs& a,
                        const CUtensorMap& tmap_act, const CUtensorMap& tmap_packed,
                        const CUtensorMap& tmap_out, int grid, cudaStream_t s);
cudaError_t launch_gemm_8bit(int mode, int bt, const GemmArgs& a, const CUtensorMap& tmap_act,
                             const CUtensorMap& tmap_packed, const CUtensorMap& tmap_out, int grid,
                             cudaStream_t s);
cudaError_t launch_gemm_f16(int mode, int bt, const GemmArgs& a, const CUtensorMap& tmap_act,
                            const CUtensorMap& tmap_packed, const CUtensorMap& tmap_out, int grid,
                            cudaStream_t s);
cudaError_t launch_splitk_reduce(const float* ws, int splits, int64_t M, int64_t ncols,
                                 void* out, int64_t ld, bool f16, cudaStream_t s);
// Bytes of the fused kernel's rings (decoded, activation and code tiles) for a
// token tile and code width: the exchange area of a cluster split (receive and
// outgoing blocks), idle once a CTA's single tile is done.
size_t gemm_exchange_bytes(int bt, int bits);
// Clusters of `cs` CTAs of the fused kernel (4-bit bf16 instance of `bt`) that can
// be resident at once on the current device; 0 when it cannot be queried.
int gemm_cluster_capacity(int mode, int bt, int cs);
// out[t] = sum over p = 0 .. P-1 in order of part[p][t] for rows inside the expert
// ranges (offsets[0] <= t < offsets[E]), 0 for the other rows of [0, T).
cudaError_t launch_row_partial_sum(const float* part, int P, int64_t T, const int32_t* offsets,
                                   int E, float* out, cudaStream_t s);

cudaError_t launch_quantize(const void* W, int w_dtype, int64_t numel, const float* code4,
                            uint8_t* packed, float* absmax, cudaStream_t s);
cudaError_t launch_quantize8(const void* W, int w_dtype, int64_t numel, const float* code,
                             uint8_t* codes, float* absmax, cudaStream_t s);
cudaError_t launch_double_quant(const float* absmax, int64_t nblocks, const float* code8,
                                uint8_t* absmax_q, float* nested_absmax, float* nested_offset,
                                double* chunk_ws, cudaStream_t s);
cudaError_t launch_dequantize(const nf4_weight& w, void* out, int out_dtype, cudaStream_t s);

constexpr int kMeanChunk = 1024;    // fixed summation order of the mean offset
constexpr int kNestedBlock = 256;   // nested blocksize

}  // namespace nf4

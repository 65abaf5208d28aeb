// nf4_gemv.cu -- small-M path of the fused NF4 products: coalesced, vectorised
// SIMT GEMV kernels with warp-shuffle reductions, for a handful of activation
// rows, where the work is bound by streaming the packed weight from HBM (Soup
// issue #842, "Design sketch": forward and transposed backward computed straight
// from the packed codes, deterministic reduction, no atomics).
//
// Both kernels read the packed codes with 16-byte loads (32 codes per lane, two
// lanes per 64-value block), decode them with the register codebook of
// decode.cuh into bf16 pairs, widen both operands exactly to fp32 and multiply
// with packed fp32x2 FMAs (fp32 accumulation).  Every sum runs in a
// fixed order: sequential within a lane, a butterfly across the warp, then warps
// (and, for the input gradient, CTAs through a workspace) in index order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "decode.cuh"
#include "internal.h"

namespace nf4 {
namespace {

constexpr int kGemvThreads = 256;  // 8 warps
constexpr int kChunk = 32;         // codes per lane per row
constexpr int kStepK = 32 * kChunk;  // 1024 k per warp and step
// weight rows per warp (forward): fewer rows when more activation rows are held
template <int MG>
struct FwdRows {
  static constexpr int value = MG <= 2 ? 2 : 1;
};
constexpr int kFwdSteps = 4;  // most contraction steps one forward warp owns
constexpr int kBwdRows = 8;        // weight rows per warp (input gradient)

// Two bf16 values (low half first) widened exactly to an fp32 pair (low word
// first) for the packed f32x2 FMA.
__device__ __forceinline__ uint64_t widen2(uint32_t v) {
  return (static_cast<uint64_t>(v & 0xFFFF0000u) << 32) | static_cast<uint64_t>(v << 16);
}

// acc.lo += a.lo * b.lo, acc.hi += a.hi * b.hi (two IEEE fp32 FMAs).
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t acc) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(acc));
  return d;
}

__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// Raw statistics of one block (absmax, or 8-bit code + nested absmax), fetched
// early; finished into the decoded scale at use.
struct Raw {
  float v;
  uint32_t q;
};

__device__ __forceinline__ Raw fetch_raw(const GemvArgs& a, int64_t n, int64_t kb) {
  const int64_t b = n * a.KB + kb;
  Raw r;
  if (!in_bounds(b >= 0 && b < a.N * a.KB, a.status)) return Raw{0.0f, 0u};  // (checked build)
  if (!a.dq) {
    r.v = __ldg(a.absmax + b);
    r.q = 0;
  } else {
    r.q = __ldg(a.absmax_q + b);
    r.v = __ldg(a.nested_absmax + (b >> 8));
  }
  return r;
}

__device__ __forceinline__ float finish(const GemvArgs& a, const Raw& r, float offset) {
  if (!a.dq) return r.v;
  return __fadd_rn(__fmul_rn(__ldg(a.code8 + r.q), r.v), offset);
}

__device__ __forceinline__ void decode32(const uint4& w4, const Lut& L, uint32_t (&o)[16]) {
  const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 d = decode8(wv[c], L);
    o[4 * c + 0] = d.x;
    o[4 * c + 1] = d.y;
    o[4 * c + 2] = d.z;
    o[4 * c + 3] = d.w;
  }
}

// Forward, activation rows m0 .. m0+MG-1.  A warp owns kFwdRows weight rows and
// up to kFwdSteps consecutive 1024-wide contraction steps; it issues all of its
// weight and statistics loads before consuming any, so the whole weight is in
// flight at once.  A CTA holds (8 / kseg) row groups; the kseg warps of a group
// split the contraction into consecutive segments, reduced in segment order.
template <int MG>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_fwd_kernel(const GemvArgs a) {
  constexpr int kFwdRows = FwdRows<MG>::value;
  constexpr int kSteps = kFwdSteps;
  __shared__ float red[8][kFwdRows][MG];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kseg = a.kseg;
  const int rg = warp / kseg, seg = warp % kseg;
  const int rows_cta = (8 / kseg) * kFwdRows;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * rows_cta + rg * kFwdRows;
  const int steps = static_cast<int>((a.K + kStepK - 1) / kStepK);
  const int s0 = seg * steps / kseg, s1 = (seg + 1) * steps / kseg;  // s1 - s0 <= kSteps
  const int64_t row_bytes = a.K / 2;

  uint4 w4[kFwdRows][kSteps];
  Raw raw[kFwdRows][kSteps];
#pragma unroll
  for (int r = 0; r < kFwdRows; ++r)
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      const int64_t n = n0 + r;
      const int64_t k = static_cast<int64_t>(s0 + i) * kStepK + lane * kChunk;
      if (s0 + i < s1 && n < a.N && k < a.K &&
          in_bounds(n >= 0 && k >= 0 && k / 2 + 16 <= row_bytes, a.status)) {
        w4[r][i] = __ldg(reinterpret_cast<const uint4*>(a.packed + n * row_bytes + k / 2));
        raw[r][i] = fetch_raw(a, n, k / 64);
      } else {
        w4[r][i] = make_uint4(0, 0, 0, 0);
        raw[r][i] = Raw{0.0f, 0u};
      }
    }
  uint64_t code2[8];
  load_code2(a.code4, code2);
  const float offset = a.dq ? __ldg(a.nested_offset) : 0.0f;

  // Accumulators hold even- and odd-indexed products of the lane's values apart
  // (one fp32 pair); they are added together after the contraction.
  uint64_t acc[kFwdRows][MG];
#pragma unroll
  for (int r = 0; r < kFwdRows; ++r)
#pragma unroll
    for (int m = 0; m < MG; ++m) acc[r][m] = 0ull;

#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int64_t k = static_cast<int64_t>(s0 + i) * kStepK + lane * kChunk;
    if (s0 + i >= s1 || k >= a.K) continue;
    uint32_t xv[MG][16];
#pragma unroll
    for (int m = 0; m < MG; ++m) {
      const uint4* xp = reinterpret_cast<const uint4*>(a.act + (a.m0 + m) * a.ld_act + k);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldg(xp + q);
        xv[m][4 * q + 0] = v.x;
        xv[m][4 * q + 1] = v.y;
        xv[m][4 * q + 2] = v.z;
        xv[m][4 * q + 3] = v.w;
      }
    }
#pragma unroll
    for (int r = 0; r < kFwdRows; ++r) {
      const Lut L = make_lut(code2, n0 + r < a.N ? finish(a, raw[r][i], offset) : 0.0f);
      uint32_t wd[16];
      decode32(w4[r][i], L, wd);
#pragma unroll
      for (int p = 0; p < 16; ++p) {
        const uint64_t wf = widen2(wd[p]);
#pragma unroll
        for (int m = 0; m < MG; ++m) acc[r][m] = fma_f32x2(wf, widen2(xv[m][p]), acc[r][m]);
      }
    }
  }
  // lanes: fixed butterfly (every lane ends with the same sum)
#pragma unroll
  for (int r = 0; r < kFwdRows; ++r)
#pragma unroll
    for (int m = 0; m < MG; ++m) {
      float v = __fadd_rn(lo_f(acc[r][m]), hi_f(acc[r][m]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp][r][m] = v;
    }
  __syncthreads();
  // segments in order
  const int t = threadIdx.x;
  if (t < rows_cta * MG) {
    const int rl = t / MG, m = t % MG;
    const int g = rl / kFwdRows, r = rl % kFwdRows;
    float v = red[g * kseg][r][m];
    for (int s = 1; s < kseg; ++s) v = __fadd_rn(v, red[g * kseg + s][r][m]);
    const int64_t n = static_cast<int64_t>(blockIdx.x) * rows_cta + rl;
    if (n < a.N && in_bounds(a.m0 + m < a.M && n < a.ld_out, a.status))
      a.out[(a.m0 + m) * a.ld_out + n] = __float2bfloat16_rn(v);
  }
}

// Input gradient, gradient rows m0 .. m0+MG-1.  CTA (kg, rgrp): k columns
// kg*1024 .. +1023 (32 per lane), weight rows rgrp*64 .. +63 (8 per warp, their
// loads issued in batches of kBwdBatch).  The 8 warps are reduced in order
// through shared memory; the CTA partial goes to ws[rgrp][m][k] (or straight to
// the output when one row group covers N).
template <int MG>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_dgrad_kernel(const GemvArgs a) {
  extern __shared__ float red[];  // [8 warps][MG][32 j][33 padded lanes]
  constexpr int kBatch = MG == 1 ? 8 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kgroups = static_cast<int>((a.K + kStepK - 1) / kStepK);
  const int kg = blockIdx.x % kgroups;
  const int64_t rgrp = blockIdx.x / kgroups;
  const int64_t k = static_cast<int64_t>(kg) * kStepK + lane * kChunk;
  const bool kvalid = k < a.K;
  const int64_t row_bytes = a.K / 2;
  const int64_t nbase = rgrp * (8 * kBwdRows) + warp * kBwdRows;

  uint64_t acc[MG][kChunk / 2];  // (value 2p, value 2p+1) of the lane's chunk
#pragma unroll
  for (int m = 0; m < MG; ++m)
#pragma unroll
    for (int j = 0; j < kChunk / 2; ++j) acc[m][j] = 0ull;

  if (kvalid) {
    uint64_t code2[8];
    load_code2(a.code4, code2);
    const float offset = a.dq ? __ldg(a.nested_offset) : 0.0f;
#pragma unroll
    for (int r0 = 0; r0 < kBwdRows; r0 += kBatch) {
      uint4 w4[kBatch];
      Raw raw[kBatch];
      uint16_t g[kBatch][MG];
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int64_t n = nbase + r0 + r;
        if (n < a.N && in_bounds(n >= 0 && k >= 0 && k / 2 + 16 <= row_bytes && a.m0 + MG <= a.M, a.status)) {
          w4[r] = __ldg(reinterpret_cast<const uint4*>(a.packed + n * row_bytes + k / 2));
          raw[r] = fetch_raw(a, n, k / 64);
#pragma unroll
          for (int m = 0; m < MG; ++m)
            g[r][m] = __ldg(reinterpret_cast<const unsigned short*>(a.act + (a.m0 + m) * a.ld_act + n));
        } else {
          w4[r] = make_uint4(0, 0, 0, 0);
          raw[r] = Raw{0.0f, 0u};
#pragma unroll
          for (int m = 0; m < MG; ++m) g[r][m] = 0;
        }
      }
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const Lut L = make_lut(code2, nbase + r0 + r < a.N ? finish(a, raw[r], offset) : 0.0f);
        uint32_t wd[16];
        decode32(w4[r], L, wd);
#pragma unroll
        for (int m = 0; m < MG; ++m) {
          const uint64_t g2 = widen2(static_cast<uint32_t>(g[r][m]) * 0x00010001u);
#pragma unroll
          for (int p = 0; p < 16; ++p) acc[m][p] = fma_f32x2(widen2(wd[p]), g2, acc[m][p]);
        }
      }
    }
  }
  // per-warp partials -> shared memory, [warp][m][j][lane] with a padded lane index
#pragma unroll
  for (int m = 0; m < MG; ++m)
#pragma unroll
    for (int p = 0; p < kChunk / 2; ++p) {
      red[((warp * MG + m) * kChunk + 2 * p) * 33 + lane] = lo_f(acc[m][p]);
      red[((warp * MG + m) * kChunk + 2 * p + 1) * 33 + lane] = hi_f(acc[m][p]);
    }
  __syncthreads();
  // warps in order; consecutive threads take consecutive k
  for (int q = threadIdx.x; q < MG * kStepK; q += kGemvThreads) {
    const int m = q / kStepK, kk = q % kStepK;
    const int ln = kk / kChunk, j = kk % kChunk;
    const int64_t kout = static_cast<int64_t>(kg) * kStepK + kk;
    if (kout >= a.K) continue;
    if (!in_bounds(a.m0 + m < a.M && kout < a.ld_out, a.status)) continue;  // (checked build)
    float v = red[((0 * MG + m) * kChunk + j) * 33 + ln];
    for (int w = 1; w < 8; ++w) v = __fadd_rn(v, red[((w * MG + m) * kChunk + j) * 33 + ln]);
    if (a.ws)
      a.ws[(rgrp * a.M + a.m0 + m) * a.K + kout] = v;
    else
      a.out[(a.m0 + m) * a.ld_out + kout] = __float2bfloat16_rn(v);
  }
}

template <int MG>
cudaError_t launch_fwd_mg(const GemvArgs& a, cudaStream_t s) {
  const int rows_cta = (8 / a.kseg) * FwdRows<MG>::value;
  const int64_t grid = (a.N + rows_cta - 1) / rows_cta;
  gemv_fwd_kernel<MG><<<static_cast<unsigned>(grid), kGemvThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int MG>
cudaError_t launch_dgrad_mg(const GemvArgs& a, int64_t rgroups, cudaStream_t s) {
  const int smem = 8 * MG * kChunk * 33 * static_cast<int>(sizeof(float));
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_dgrad_kernel<MG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t kgroups = (a.K + kStepK - 1) / kStepK;
  gemv_dgrad_kernel<MG><<<static_cast<unsigned>(kgroups * rgroups), kGemvThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int gemv_fwd_kseg(int64_t K) {
  // segments of at most kFwdSteps steps; a power of two dividing the 8 warps
  const int64_t steps = (K + kStepK - 1) / kStepK;
  int kseg = 1;
  while (kseg < 8 && (steps + kseg - 1) / kseg > kFwdSteps) kseg *= 2;
  return kseg;
}

int64_t gemv_dgrad_row_groups(int64_t N) { return (N + 8 * kBwdRows - 1) / (8 * kBwdRows); }

cudaError_t launch_gemv_fwd(const GemvArgs& a0, cudaStream_t s) {
  // activation rows in groups of at most 4 (each group re-reads the weight)
  for (int m0 = 0; m0 < a0.M; m0 += 4) {
    GemvArgs a = a0;
    a.m0 = m0;
    const int mg = a0.M - m0 < 4 ? static_cast<int>(a0.M - m0) : 4;
    cudaError_t e;
    switch (mg) {
      case 1: e = launch_fwd_mg<1>(a, s); break;
      case 2: e = launch_fwd_mg<2>(a, s); break;
      case 3: e = launch_fwd_mg<3>(a, s); break;
      default: e = launch_fwd_mg<4>(a, s); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gemv_dgrad(const GemvArgs& a0, cudaStream_t s) {
  const int64_t rgroups = gemv_dgrad_row_groups(a0.N);
  for (int m0 = 0; m0 < a0.M; m0 += 2) {
    GemvArgs a = a0;
    a.m0 = m0;
    if (rgroups == 1) a.ws = nullptr;
    const int mg = a0.M - m0 < 2 ? 1 : 2;
    cudaError_t e = mg == 1 ? launch_dgrad_mg<1>(a, rgroups, s) : launch_dgrad_mg<2>(a, rgroups, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace nf4

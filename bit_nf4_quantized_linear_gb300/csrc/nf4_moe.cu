// nf4_moe.cu -- the top-k combine of the grouped experts and its backward.
//
// The grouped products leave one output row per (token, routed expert), sorted by
// expert (fork PR "Experts trainability", commits 1-2: per-expert segments; Soup
// issue #842, expert path).  The combine gives each token the sum of its routed
// rows, the routing weights having been applied in the down projection's
// epilogue (row scale):
//   out[t][c] = bf16( sum_{j = 0 .. k-1, token_rows[t][j] >= 0} rows[token_rows[t][j]][c] )
// with the sum in fp32 in route order j (deterministic, no atomics).  Its
// backward copies each token's gradient to the rows it was routed to:
//   grad_rows[token_rows[t][j]] = grad_out[t].
// Both kernels move 16-byte vectors (8 bf16) and are bound by HBM; a route index
// outside [0, R) is skipped and recorded as NF4_ERR_BAD_OFFSETS.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace nf4 {
namespace {

constexpr int kMoeThreads = 256;
constexpr int kMoeCols = kMoeThreads * 8;  // columns per CTA (8 per thread)

__device__ __forceinline__ void add8(float (&acc)[8], const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(w[i] << 16));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(w[i] & 0xffff0000u));
  }
}

// One CTA per (token, chunk of kMoeCols columns): blockIdx.x the token,
// blockIdx.y the chunk.
__global__ void __launch_bounds__(kMoeThreads) moe_combine_kernel(MoeArgs a) {
  const int64_t t = blockIdx.x;
  const int64_t c = static_cast<int64_t>(blockIdx.y) * kMoeCols + threadIdx.x * 8;
  if (c >= a.H) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // Eight routes at a time: their indices, then all their row loads in flight
  // together, then the adds in route order (an absent route, -1, is skipped).
  for (int j0 = 0; j0 < a.k; j0 += 8) {
    int32_t rr[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) rr[u] = j0 + u < a.k ? a.token_rows[t * a.k + j0 + u] : -1;
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool ok = rr[u] >= 0 && rr[u] < a.R;
      if (rr[u] >= a.R && a.status) atomicCAS(a.status, 0, NF4_ERR_BAD_OFFSETS);
      v[u] = ok ? *reinterpret_cast<const uint4*>(a.rows + static_cast<int64_t>(rr[u]) * a.ld_rows + c)
                : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (rr[u] >= 0 && rr[u] < a.R) add8(acc, v[u]);
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(a.out + t * a.ld_out + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Backward: grad_out[t] to each row token t was routed to.
__global__ void __launch_bounds__(kMoeThreads) moe_combine_bwd_kernel(MoeArgs a) {
  const int64_t t = blockIdx.x;
  const int64_t c = static_cast<int64_t>(blockIdx.y) * kMoeCols + threadIdx.x * 8;
  if (c >= a.H) return;
  const uint4 g = *reinterpret_cast<const uint4*>(a.rows + t * a.ld_rows + c);
  for (int j = 0; j < a.k; ++j) {
    const int32_t r = a.token_rows[t * a.k + j];
    if (r < 0) continue;
    if (r >= a.R) {
      if (a.status) atomicCAS(a.status, 0, NF4_ERR_BAD_OFFSETS);
      continue;
    }
    *reinterpret_cast<uint4*>(a.out + static_cast<int64_t>(r) * a.ld_out + c) = g;
  }
}

}  // namespace

cudaError_t launch_moe(bool backward, const MoeArgs& a, cudaStream_t s) {
  if (a.tokens == 0 || a.H == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(a.tokens), static_cast<unsigned>((a.H + kMoeCols - 1) / kMoeCols), 1);
  if (backward)
    moe_combine_bwd_kernel<<<grid, kMoeThreads, 0, s>>>(a);
  else
    moe_combine_kernel<<<grid, kMoeThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace nf4

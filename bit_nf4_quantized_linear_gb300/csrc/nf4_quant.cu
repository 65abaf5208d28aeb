// nf4_quant.cu -- blockwise NF4 (and 8-bit) quantisation, with double
// quantisation of the absmax statistics, and dense dequantisation.
//
// quantize_4bit(w, blocksize=64, quant_type="nf4", compress_statistics=True) and
// dequantize_4bit(B, state) of bitsandbytes issue "MatMul4Bit keeps B and
// quant_state on ctx ..." (sections "Minimal reproducer" and "Root cause").  These
// steps are offline (quantisation) or off the fused path (dense dequantisation);
// both are bit-exact with the CPU reference because every floating-point step is
// one IEEE-rounded operation written with an explicit rounding intrinsic:
//   - normalisation v = w / absmax by IEEE division (__fdiv_rn);
//   - nearest level by comparison with fp64 midpoints of adjacent levels, an exact
//     tie going to the lower index;
//   - the mean offset summed in fp64 over chunks of 1024 values, then over the
//     chunk sums in order, divided in fp64 and rounded once to fp32;
//   - decoded scale fp32(fp32(code8[q]*na) + offset) with two roundings, no FMA.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace nf4 {
namespace {

// Count of midpoints strictly below v; midpoints are ascending.
__device__ __forceinline__ int count_below(const double* mid, int nmid, float v) {
  const double dv = static_cast<double>(v);
  int lo = 0, hi = nmid;  // first index with mid >= v
  while (lo < hi) {
    int m = (lo + hi) >> 1;
    if (mid[m] < dv) lo = m + 1; else hi = m;
  }
  return lo;
}

template <typename T>
__device__ __forceinline__ float load_as_f32(const T* p, int64_t i);
template <>
__device__ __forceinline__ float load_as_f32<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_as_f32<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);  // exact widening
}

// One warp per block of 64 values; lane l owns values 2l and 2l+1 of the block.
template <typename T>
__global__ void __launch_bounds__(256) quantize_blocks_kernel(const T* __restrict__ W, int64_t numel,
                                                               const float* __restrict__ code4,
                                                               uint8_t* __restrict__ packed,
                                                               float* __restrict__ absmax) {
  __shared__ double mid[15];
  __shared__ int zero_idx;
  if (threadIdx.x < 15)
    mid[threadIdx.x] = __dmul_rn(__dadd_rn(static_cast<double>(code4[threadIdx.x]),
                                           static_cast<double>(code4[threadIdx.x + 1])), 0.5);
  if (threadIdx.x == 0) {
    int z = 0;
    for (int j = 15; j >= 0; --j)
      if (code4[j] == 0.0f) z = j;
    zero_idx = z;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int64_t nblocks = (numel + 63) / 64;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t blk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       blk < nblocks; blk += warps_total) {
    const int64_t e0 = blk * 64 + 2 * lane;
    const bool has0 = e0 < numel, has1 = e0 + 1 < numel;
    const float v0 = has0 ? load_as_f32(W, e0) : 0.0f;
    const float v1 = has1 ? load_as_f32(W, e0 + 1) : 0.0f;
    float a = fmaxf(has0 ? fabsf(v0) : 0.0f, has1 ? fabsf(v1) : 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) absmax[blk] = a;
    int q0 = 0, q1 = 0;
    if (a == 0.0f) {
      q0 = zero_idx;
      q1 = has1 ? zero_idx : 0;
    } else {
      q0 = count_below(mid, 15, __fdiv_rn(v0, a));
      q1 = has1 ? count_below(mid, 15, __fdiv_rn(v1, a)) : 0;
    }
    if (has0) packed[e0 >> 1] = static_cast<uint8_t>((q0 << 4) | q1);
  }
}

// 8-bit storage (one code per byte, 256-level codebook): the same block steps as
// above.  One warp per block of 64 values; lane l owns values 2l and 2l+1.
template <typename T>
__global__ void __launch_bounds__(256) quantize8_blocks_kernel(const T* __restrict__ W, int64_t numel,
                                                                const float* __restrict__ code,
                                                                uint8_t* __restrict__ codes,
                                                                float* __restrict__ absmax) {
  __shared__ double mid[255];
  __shared__ int zero_idx;
  for (int j = threadIdx.x; j < 255; j += blockDim.x)
    mid[j] = __dmul_rn(__dadd_rn(static_cast<double>(code[j]), static_cast<double>(code[j + 1])), 0.5);
  if (threadIdx.x == 0) {
    int z = 0;
    for (int j = 255; j >= 0; --j)
      if (code[j] == 0.0f) z = j;
    zero_idx = z;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int64_t nblocks = (numel + 63) / 64;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t blk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       blk < nblocks; blk += warps_total) {
    const int64_t e0 = blk * 64 + 2 * lane;
    const bool has0 = e0 < numel, has1 = e0 + 1 < numel;
    const float v0 = has0 ? load_as_f32(W, e0) : 0.0f;
    const float v1 = has1 ? load_as_f32(W, e0 + 1) : 0.0f;
    float a = fmaxf(has0 ? fabsf(v0) : 0.0f, has1 ? fabsf(v1) : 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) absmax[blk] = a;
    const int q0 = a == 0.0f ? zero_idx : count_below(mid, 255, __fdiv_rn(v0, a));
    const int q1 = a == 0.0f ? zero_idx : count_below(mid, 255, __fdiv_rn(v1, a));
    if (has0) codes[e0] = static_cast<uint8_t>(q0);
    if (has1) codes[e0 + 1] = static_cast<uint8_t>(q1);
  }
}

// fp64 sum of each chunk of kMeanChunk absmax values, sequential within the chunk.
__global__ void chunk_sum_kernel(const float* __restrict__ absmax, int64_t nblocks,
                                 double* __restrict__ chunk) {
  const int64_t nchunks = (nblocks + kMeanChunk - 1) / kMeanChunk;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunks;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b0 = c * kMeanChunk;
    const int64_t b1 = b0 + kMeanChunk < nblocks ? b0 + kMeanChunk : nblocks;
    double s = 0.0;
    for (int64_t b = b0; b < b1; ++b) s = __dadd_rn(s, static_cast<double>(absmax[b]));
    chunk[c] = s;
  }
}

// Sequential sum of the chunk sums; the mean rounded once to fp32.
__global__ void mean_offset_kernel(const double* __restrict__ chunk, int64_t nblocks,
                                   float* __restrict__ offset) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const int64_t nchunks = (nblocks + kMeanChunk - 1) / kMeanChunk;
  double total = 0.0;
  for (int64_t c = 0; c < nchunks; ++c) total = __dadd_rn(total, chunk[c]);
  *offset = __double2float_rn(__ddiv_rn(total, static_cast<double>(nblocks)));
}

// One CTA of 256 threads per nested block of 256 absmax values.
__global__ void __launch_bounds__(kNestedBlock) nested_quant_kernel(
    const float* __restrict__ absmax, int64_t nblocks, const float* __restrict__ code8,
    const float* __restrict__ offset, uint8_t* __restrict__ absmax_q,
    float* __restrict__ nested_absmax) {
  __shared__ double mid[255];
  __shared__ float red[kNestedBlock / 32];
  __shared__ int zero_idx;
  for (int j = threadIdx.x; j < 255; j += blockDim.x)
    mid[j] = __dmul_rn(__dadd_rn(static_cast<double>(code8[j]), static_cast<double>(code8[j + 1])), 0.5);
  if (threadIdx.x == 0) {
    int z = 0;
    for (int j = 255; j >= 0; --j)
      if (code8[j] == 0.0f) z = j;
    zero_idx = z;
  }
  const float off = *offset;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kNestedBlock + threadIdx.x;
  const bool has = b < nblocks;
  const float r = has ? __fsub_rn(absmax[b], off) : 0.0f;
  float m = fabsf(r);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  float na = 0.0f;
#pragma unroll
  for (int w = 0; w < kNestedBlock / 32; ++w) na = fmaxf(na, red[w]);
  if (threadIdx.x == 0) nested_absmax[blockIdx.x] = na;
  if (has) {
    int q = (na == 0.0f) ? zero_idx : count_below(mid, 255, __fdiv_rn(r, na));
    absmax_q[b] = static_cast<uint8_t>(q);
  }
}

__device__ __forceinline__ float block_scale(const nf4_weight& w, int64_t b,
                                             const float* code8_s) {
  if (!w.double_quant) return w.absmax[b];
  const float t = __fmul_rn(code8_s[w.absmax_q[b]], w.nested_absmax[b / kNestedBlock]);
  return __fadd_rn(t, *w.nested_offset);
}

// One thread per packed byte (two values).
template <typename OutT>
__global__ void __launch_bounds__(256) dequantize_kernel(nf4_weight w, int64_t numel, OutT* __restrict__ out) {
  __shared__ float code4_s[16];
  __shared__ float code8_s[256];
  if (threadIdx.x < 16) code4_s[threadIdx.x] = w.code4[threadIdx.x];
  if (w.double_quant)
    for (int j = threadIdx.x; j < 256; j += blockDim.x) code8_s[j] = w.code8[j];
  __syncthreads();
  const int64_t nbytes = (numel + 1) / 2;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < nbytes;
       j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint8_t byte = w.packed[j];
    const int64_t i0 = 2 * j;
    const float s0 = block_scale(w, i0 / w.blocksize, code8_s);
    const float f0 = __fmul_rn(code4_s[byte >> 4], s0);
    if constexpr (sizeof(OutT) == 4) out[i0] = f0;
    else out[i0] = __float2bfloat16_rn(f0);
    if (i0 + 1 < numel) {
      const float s1 = block_scale(w, (i0 + 1) / w.blocksize, code8_s);
      const float f1 = __fmul_rn(code4_s[byte & 15], s1);
      if constexpr (sizeof(OutT) == 4) out[i0 + 1] = f1;
      else out[i0 + 1] = __float2bfloat16_rn(f1);
    }
  }
}

// 8-bit storage: one thread per value.
template <typename OutT>
__global__ void __launch_bounds__(256) dequantize8_kernel(nf4_weight w, int64_t numel, OutT* __restrict__ out) {
  __shared__ float code_s[256];
  __shared__ float code8_s[256];
  for (int j = threadIdx.x; j < 256; j += blockDim.x) {
    code_s[j] = w.code4[j];
    if (w.double_quant) code8_s[j] = w.code8[j];
  }
  __syncthreads();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < numel;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float f = __fmul_rn(code_s[w.packed[i]], block_scale(w, i / w.blocksize, code8_s));
    if constexpr (sizeof(OutT) == 4) out[i] = f;
    else out[i] = __float2bfloat16_rn(f);
  }
}

int grid_for(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 65535 * 16) g = 65535 * 16;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_quantize(const void* W, int w_dtype, int64_t numel, const float* code4,
                            uint8_t* packed, float* absmax, cudaStream_t s) {
  const int64_t nblocks = (numel + 63) / 64;
  const int grid = grid_for(nblocks, 8);
  if (w_dtype == NF4_DTYPE_F32)
    quantize_blocks_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(W), numel, code4,
                                                        packed, absmax);
  else
    quantize_blocks_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(W), numel, code4, packed, absmax);
  return cudaGetLastError();
}

cudaError_t launch_quantize8(const void* W, int w_dtype, int64_t numel, const float* code,
                             uint8_t* codes, float* absmax, cudaStream_t s) {
  const int64_t nblocks = (numel + 63) / 64;
  const int grid = grid_for(nblocks, 8);
  if (w_dtype == NF4_DTYPE_F32)
    quantize8_blocks_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(W), numel, code,
                                                         codes, absmax);
  else
    quantize8_blocks_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(W), numel, code, codes, absmax);
  return cudaGetLastError();
}

cudaError_t launch_double_quant(const float* absmax, int64_t nblocks, const float* code8,
                                uint8_t* absmax_q, float* nested_absmax, float* nested_offset,
                                double* chunk_ws, cudaStream_t s) {
  const int64_t nchunks = (nblocks + kMeanChunk - 1) / kMeanChunk;
  chunk_sum_kernel<<<grid_for(nchunks, 128), 128, 0, s>>>(absmax, nblocks, chunk_ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mean_offset_kernel<<<1, 32, 0, s>>>(chunk_ws, nblocks, nested_offset);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nnested = (nblocks + kNestedBlock - 1) / kNestedBlock;
  nested_quant_kernel<<<static_cast<unsigned>(nnested), kNestedBlock, 0, s>>>(
      absmax, nblocks, code8, nested_offset, absmax_q, nested_absmax);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const nf4_weight& w, void* out, int out_dtype, cudaStream_t s) {
  const int64_t numel = w.N * w.K;
  if (w.bits == 8) {
    const int grid8 = grid_for(numel, 256 * 4);
    if (out_dtype == NF4_DTYPE_F32)
      dequantize8_kernel<float><<<grid8, 256, 0, s>>>(w, numel, static_cast<float*>(out));
    else
      dequantize8_kernel<__nv_bfloat16><<<grid8, 256, 0, s>>>(w, numel, static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError();
  }
  const int grid = grid_for((numel + 1) / 2, 256 * 4);
  if (out_dtype == NF4_DTYPE_F32)
    dequantize_kernel<float><<<grid, 256, 0, s>>>(w, numel, static_cast<float*>(out));
  else
    dequantize_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(w, numel, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace nf4

// decode.cuh -- register-resident NF4 codebook decode shared by the fused kernels.
//
// A 64-value block of packed 4-bit codes and its scale s become bf16 values
// bf16(fp32(code4[q] * s)) (bitsandbytes issue "MatMul4Bit keeps B and
// quant_state on ctx ...", "Root cause": dequantize_4bit), computed without a
// per-value multiply: the 16 scaled codebook entries are built once per block and
// looked up four at a time with byte permutes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace nf4 {

// The 16 bf16 values T[q] = bf16(fp32(code4[q] * s)) of one 64-value block,
// held in registers as byte planes: lo[k] packs the low bytes of T[4k..4k+3],
// hi[k] the high bytes.  A byte permute (prmt) then looks up four codes at once.
struct Lut {
  uint32_t lo[4], hi[4];
};

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));  // two IEEE products
  return d;
}

// Two fp32 values to a pair of 16-bit floats (the first in the low half), round to
// nearest even: bf16, or IEEE fp16 when F16.
template <bool F16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
  }
}

// code2[i] holds code4[2i] (low word) and code4[2i+1] (high word).  Entries are
// bf16 (or fp16 when F16) of fp32(code4[q] * s).
template <bool F16 = false>
__device__ __forceinline__ Lut make_lut(const uint64_t (&code2)[8], float s) {
  const uint64_t s2 = (static_cast<uint64_t>(__float_as_uint(s)) << 32) | __float_as_uint(s);
  uint32_t p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t m = mul_f32x2(code2[i], s2);
    p[i] = pack16x2<F16>(__uint_as_float(static_cast<uint32_t>(m)),  // T[2i] low half,
                         __uint_as_float(static_cast<uint32_t>(m >> 32)));  // T[2i+1] high half
  }
  Lut L;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    L.lo[k] = __byte_perm(p[2 * k], p[2 * k + 1], 0x6420u);
    L.hi[k] = __byte_perm(p[2 * k], p[2 * k + 1], 0x7531u);
  }
  return L;
}

// Four codes (the low 16 bits of v) to the byte planes of their bf16 values:
// byte i of `lo` / `hi` is the low / high byte of T[code in nibble position i].
__device__ __forceinline__ void planes4(uint32_t v, const Lut& L, uint32_t& lo, uint32_t& hi) {
  const uint32_t sel = v & 0x7777u;                      // low 3 bits of each code
  const uint32_t s3 = ((v >> 1) & 0x4444u) | 0x3210u;   // code bit 3 picks the upper 8 entries
  lo = __byte_perm(__byte_perm(L.lo[0], L.lo[1], sel), __byte_perm(L.lo[2], L.lo[3], sel), s3);
  hi = __byte_perm(__byte_perm(L.hi[0], L.hi[1], sel), __byte_perm(L.hi[2], L.hi[3], sel), s3);
}

// Four codes (the low 16 bits of v: nibble positions 0..3 = values 1, 0, 3, 2 of a
// byte pair, even value in the high nibble) to two bf16 pairs, value 0 lowest.
__device__ __forceinline__ void lookup4(uint32_t v, const Lut& L, uint32_t& out01,
                                        uint32_t& out23) {
  uint32_t lo, hi;
  planes4(v, L, lo, hi);
  out01 = __byte_perm(lo, hi, 0x4051u);
  out23 = __byte_perm(lo, hi, 0x6273u);
}

// Eight packed codes (one 32-bit word; byte j holds value 2j high, 2j+1 low) to
// eight bf16 values, packed pairwise, value 0 lowest.  The permute selectors of
// both halves come from one mask of the whole word (a permute reads only the low
// 16 bits of its selector).
__device__ __forceinline__ uint4 decode8(uint32_t w, const Lut& L) {
  const uint32_t sel = w & 0x77777777u;
  const uint32_t s3 = ((w >> 1) & 0x44444444u) | 0x32103210u;
  const uint32_t sel_h = sel >> 16, s3_h = s3 >> 16;
  uint4 o;
  uint32_t lo = __byte_perm(__byte_perm(L.lo[0], L.lo[1], sel), __byte_perm(L.lo[2], L.lo[3], sel), s3);
  uint32_t hi = __byte_perm(__byte_perm(L.hi[0], L.hi[1], sel), __byte_perm(L.hi[2], L.hi[3], sel), s3);
  o.x = __byte_perm(lo, hi, 0x4051u);
  o.y = __byte_perm(lo, hi, 0x6273u);
  lo = __byte_perm(__byte_perm(L.lo[0], L.lo[1], sel_h), __byte_perm(L.lo[2], L.lo[3], sel_h), s3_h);
  hi = __byte_perm(__byte_perm(L.hi[0], L.hi[1], sel_h), __byte_perm(L.hi[2], L.hi[3], sel_h), s3_h);
  o.z = __byte_perm(lo, hi, 0x4051u);
  o.w = __byte_perm(lo, hi, 0x6273u);
  return o;
}


// code2[i] = (code4[2i+1] << 32) | code4[2i] from a 16-entry fp32 codebook.
__device__ __forceinline__ void load_code2(const float* code4, uint64_t (&code2)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    code2[i] = (static_cast<uint64_t>(__float_as_uint(code4[2 * i + 1])) << 32) |
               __float_as_uint(code4[2 * i]);
}

}  // namespace nf4

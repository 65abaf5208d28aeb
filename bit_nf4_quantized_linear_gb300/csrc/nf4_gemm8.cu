// nf4_gemm8.cu -- the fused kernel's instances for 8-bit codes (one code per byte,
// 256-level codebook; blockwise int8 dynamic map or e4m3 levels), compiled as a
// separate translation unit so the two code widths build in parallel.
#define NF4_GEMM_BITS 8
#include "nf4_gemm.cu"

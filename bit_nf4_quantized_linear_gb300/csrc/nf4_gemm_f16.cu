// nf4_gemm_f16.cu -- the fused kernel's instances for the fp16 compute dtype
// (fp16 activations, fp16 dequantised operand, fp16 output; 4-bit codes), compiled
// as a separate translation unit so the variants build in parallel.
#define NF4_GEMM_BITS 4
#define NF4_GEMM_F16 1
#include "nf4_gemm.cu"

// kern_tf32_bf16.cu -- tcgen05 GEMM kernels with FP32 inputs used as TF32
// (kind::tf32) and bf16 output.
#define KERN_OUT_T __nv_bfloat16
#define KERN_SUFFIX tf32_bf16
#define KERN_ES 4
#include "kern_inst.cuh"

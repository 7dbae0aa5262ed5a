// kern_bf16.cu -- tcgen05 GEMM kernels with bf16 output.
#define KERN_OUT_T __nv_bfloat16
#define KERN_SUFFIX bf16
#define KERN_ES 2
#include "kern_inst.cuh"

// kern_tf32_f16.cu -- tcgen05 GEMM kernels with FP32 inputs used as TF32
// (kind::tf32) and f16 output.
#define KERN_OUT_T __half
#define KERN_SUFFIX tf32_f16
#define KERN_ES 4
#include "kern_inst.cuh"

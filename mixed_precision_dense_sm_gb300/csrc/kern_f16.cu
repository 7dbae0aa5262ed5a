// kern_f16.cu -- tcgen05 GEMM kernels with f16 output.
#define KERN_OUT_T __half
#define KERN_SUFFIX f16
#define KERN_ES 2
#include "kern_inst.cuh"

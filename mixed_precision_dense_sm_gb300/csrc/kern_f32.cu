// kern_f32.cu -- tcgen05 GEMM kernels with f32 output.
#define KERN_OUT_T float
#define KERN_SUFFIX f32
#define KERN_ES 2
#include "kern_inst.cuh"

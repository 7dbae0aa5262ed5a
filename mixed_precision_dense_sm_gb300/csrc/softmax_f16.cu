// softmax_f16.cu -- row-softmax kernels with f16 input, every output type.
#define SMX_IN_T __half
#define SMX_SUFFIX f16
#include "softmax_inst.cuh"

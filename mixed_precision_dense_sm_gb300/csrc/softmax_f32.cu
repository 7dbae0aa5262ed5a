// softmax_f32.cu -- row-softmax kernels with f32 input, every output type.
#define SMX_IN_T float
#define SMX_SUFFIX f32
#include "softmax_inst.cuh"

// softmax_bf16.cu -- row-softmax kernels with bf16 input, every output type.
#define SMX_IN_T __nv_bfloat16
#define SMX_SUFFIX bf16
#include "softmax_inst.cuh"

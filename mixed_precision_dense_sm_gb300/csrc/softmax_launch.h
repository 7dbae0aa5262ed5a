// softmax_launch.h -- internal interface between the softmax host code
// (softmax.cu) and the translation units that instantiate the kernel for each
// input type (softmax_{f32,f16,bf16}.cu).  Output type codes follow
// gemm_dtype_t: 0 = F16, 1 = BF16, 2 = F32.
#pragma once
#include <cuda_runtime.h>

#include "softmax_kern.cuh"
#include "softmax_tma.cuh"

namespace smx {

#define SMX_DECLARE(suffix)                                                                 \
    cudaError_t launch_softmax_##suffix(const SoftmaxParams& p, int y_dtype, bool warp_rows,  \
                                        int threads, int grid, cudaStream_t stream);         \
    int resident_groups_##suffix(int y_dtype, bool warp_rows, int threads, int cluster,      \
                                 int num_sms);                                               \
    cudaError_t launch_softmax_tma_##suffix(const TmaSoftmaxParams& p, int y_dtype, int grid, \
                                            size_t smem, cudaStream_t stream);
SMX_DECLARE(f32)
SMX_DECLARE(f16)
SMX_DECLARE(bf16)
#undef SMX_DECLARE

}  // namespace smx

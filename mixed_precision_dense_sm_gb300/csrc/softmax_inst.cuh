// softmax_inst.cuh -- instantiates the row-softmax kernel for one input type
// (SMX_IN_T) and every output type, behind plain launchers.
#pragma once
#include "softmax_launch.h"

#define SMX_CAT2(a, b) a##b
#define SMX_CAT(a, b) SMX_CAT2(a, b)

namespace smx {

cudaError_t SMX_CAT(launch_softmax_, SMX_SUFFIX)(const SoftmaxParams& p, int y_dtype,
                                                 bool warp_rows, int threads, int grid,
                                                 cudaStream_t stream) {
    switch (y_dtype) {
        case 0: return launch_softmax<SMX_IN_T, __half>(p, warp_rows, threads, grid, stream);
        case 1: return launch_softmax<SMX_IN_T, __nv_bfloat16>(p, warp_rows, threads, grid, stream);
        case 2: return launch_softmax<SMX_IN_T, float>(p, warp_rows, threads, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t SMX_CAT(launch_softmax_tma_, SMX_SUFFIX)(const TmaSoftmaxParams& p, int y_dtype,
                                                     int grid, size_t smem, cudaStream_t stream) {
    switch (y_dtype) {
        case 0: return launch_softmax_tma<SMX_IN_T, __half>(p, grid, smem, stream);
        case 1: return launch_softmax_tma<SMX_IN_T, __nv_bfloat16>(p, grid, smem, stream);
        case 2: return launch_softmax_tma<SMX_IN_T, float>(p, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

int SMX_CAT(resident_groups_, SMX_SUFFIX)(int y_dtype, bool warp_rows, int threads, int cluster,
                                          int num_sms) {
    switch (y_dtype) {
        case 0: return resident_groups<SMX_IN_T, __half>(warp_rows, threads, cluster, num_sms);
        case 1: return resident_groups<SMX_IN_T, __nv_bfloat16>(warp_rows, threads, cluster, num_sms);
        default: return resident_groups<SMX_IN_T, float>(warp_rows, threads, cluster, num_sms);
    }
}

}  // namespace smx

// kern_inst.cuh -- instantiates the tcgen05 GEMM and its stream-K fixup for one
// output type (KERN_OUT_T) and the three tile widths, behind plain launchers.
#pragma once
#include "launch.h"

#define GEMM103_CAT2(a, b) a##b
#define GEMM103_CAT(a, b) GEMM103_CAT2(a, b)

namespace gemm103 {

template <int BN>
static cudaError_t launch_tc_bn(const TcLaunch& l) {
    auto kern = gemm_tc_kernel<BN, KERN_OUT_T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(l.smem_bytes));
    if (e != cudaSuccess) return e;
    kern<<<l.grid, kThreads, l.smem_bytes, l.stream>>>(l.tmA, l.tmB, l.p);
    return cudaGetLastError();
}

cudaError_t GEMM103_CAT(launch_tc_, KERN_SUFFIX)(const TcLaunch& l) {
    switch (l.block_n) {
        case 64: return launch_tc_bn<64>(l);
        case 128: return launch_tc_bn<128>(l);
        case 256: return launch_tc_bn<256>(l);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t GEMM103_CAT(launch_fixup_, KERN_SUFFIX)(const TcLaunch& l, int grid) {
    switch (l.block_n) {
        case 64: streamk_fixup_kernel<64, KERN_OUT_T><<<grid, 256, 0, l.stream>>>(l.p); break;
        case 128: streamk_fixup_kernel<128, KERN_OUT_T><<<grid, 256, 0, l.stream>>>(l.p); break;
        case 256: streamk_fixup_kernel<256, KERN_OUT_T><<<grid, 256, 0, l.stream>>>(l.p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gemm103

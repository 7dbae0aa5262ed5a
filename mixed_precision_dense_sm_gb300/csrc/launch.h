// launch.h -- internal interface between the host planner (api.cu) and the
// translation units that instantiate the kernels for each output type.
#pragma once
#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_tc.cuh"

namespace gemm103 {

struct TcLaunch {
    CUtensorMap tmA, tmB;
    CUtensorMap tmC;    // C for the epilogue's TMA stores (p.c_tma), else unused
    TcParams p;
    int grid;
    int cta_group;      // 1: single-CTA tiles, 2: CTA-pair tiles
    int block_n;
    int esize;          // input element bytes: 2 (FP16/BF16) or 4 (FP32 used as TF32)
    int epi;            // kEpiPlain or kEpiLayerNorm (16-bit inputs only)
    int kc;             // K chunks per stage: 1, or 2 (tiles whose 3 stages fit)
    int mh;             // M halves per single-CTA tile: 1 (128 rows) or 2 (256 rows, BN <= 128)
    size_t smem_bytes;
    cudaStream_t stream;
};

// One launcher per (input element size, output type); the output type codes
// follow gemm_dtype_t: 0 = F16, 1 = BF16, 2 = F32.
cudaError_t launch_tc_f32(const TcLaunch& l);
cudaError_t launch_tc_f16(const TcLaunch& l);
cudaError_t launch_tc_bf16(const TcLaunch& l);
cudaError_t launch_tc_tf32_f32(const TcLaunch& l);
cudaError_t launch_tc_tf32_f16(const TcLaunch& l);
cudaError_t launch_tc_tf32_bf16(const TcLaunch& l);

}  // namespace gemm103

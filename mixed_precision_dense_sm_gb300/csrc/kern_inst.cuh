// kern_inst.cuh -- instantiates the tcgen05 GEMM for one input element size
// (KERN_ES bytes: 2 for FP16/BF16, 4 for FP32 used as TF32) and one output
// type (KERN_OUT_T): single-CTA tiles of width 64/128/256 and CTA-pair tiles
// of width 256, behind a plain launcher -- and, for 16-bit inputs, the
// LayerNorm-epilogue variants (single-CTA 128/256, CTA-pair 256) and the
// 256-row single-CTA tiles of width 64/128 (MH = 2, used by convolutions).  Each with
// one K chunk per stage, and those whose three stages of two chunks fit in
// shared memory also with two; the plain single-CTA 256-wide tile also with
// two (two stages, used by convolutions).
#pragma once
#include <mutex>

#include "launch.h"

#define GEMM103_CAT2(a, b) a##b
#define GEMM103_CAT(a, b) GEMM103_CAT2(a, b)

namespace gemm103 {

template <int CG, int BN, int EPI = kEpiPlain, int KC = 1, int MH = 1>
static cudaError_t launch_tc_cfg(const TcLaunch& l) {
    auto kern = gemm_tc_kernel<CG, BN, KERN_OUT_T, KERN_ES, EPI, KC, MH>;
    {
        // The dynamic shared-memory limit is raised once per size (a host
        // call worth avoiding on every launch of a microsecond-scale GEMM).
        static std::mutex mu;
        static size_t raised_to = 0;
        std::lock_guard<std::mutex> g(mu);
        if (l.smem_bytes > raised_to) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(l.smem_bytes));
            if (e != cudaSuccess) return e;
            raised_to = l.smem_bytes;
        }
    }
    // Programmatic stream serialisation: the kernel's set-up may overlap the
    // tail of the previous kernel on the stream (the kernel waits for it with
    // griddepcontrol.wait before touching global memory).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = l.smem_bytes;
    cfg.stream = l.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (CG == 1) {
        cfg.gridDim = dim3(l.grid, 1, 1);
        return cudaLaunchKernelEx(&cfg, kern, l.tmA, l.tmB, l.tmC, l.p);
    } else {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        int grid = l.grid;
        if (!l.p.stream_k) {
            // A data-parallel schedule adapts to the grid: launch no more
            // pairs than can be resident at once (persistent CTAs).
            static std::mutex mu;
            static size_t cached_smem = 0;
            static int cached_clusters = 0;
            int clusters = 0;
            {
                std::lock_guard<std::mutex> g(mu);
                if (cached_smem != l.smem_bytes) {
                    // the query takes the cluster shape alone
                    cudaLaunchConfig_t q = cfg;
                    q.gridDim = dim3(grid, 1, 1);
                    q.attrs = &attr[1];
                    q.numAttrs = 1;
                    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &q) != cudaSuccess) {
                        cudaGetLastError();
                        clusters = 0;
                    }
                    cached_smem = l.smem_bytes;
                    cached_clusters = clusters;
                }
                clusters = cached_clusters;
            }
            if (clusters > 0 && grid > 2 * clusters) grid = 2 * clusters;
        }
        cfg.gridDim = dim3(grid, 1, 1);
        return cudaLaunchKernelEx(&cfg, kern, l.tmA, l.tmB, l.tmC, l.p);
    }
}

template <int KC>
static cudaError_t launch_tc_kc(const TcLaunch& l) {
    if (l.epi == kEpiLayerNorm) {
        if constexpr (KERN_ES == 2) {
            if (l.cta_group == 2)
                return l.block_n == 256 ? launch_tc_cfg<2, 256, kEpiLayerNorm, KC>(l)
                                        : cudaErrorInvalidValue;
            switch (l.block_n) {
                case 128: return launch_tc_cfg<1, 128, kEpiLayerNorm, KC>(l);
                case 256:
                    if constexpr (KC == 1) return launch_tc_cfg<1, 256, kEpiLayerNorm, 1>(l);
                    return cudaErrorInvalidValue;
                default: return cudaErrorInvalidValue;
            }
        }
        return cudaErrorInvalidValue;
    }
    if (l.epi != kEpiPlain) return cudaErrorInvalidValue;
    if (l.mh == 2) {
        // 256-row single-CTA tiles (16-bit inputs: convolutions)
        if constexpr (KERN_ES == 2) {
            if (l.cta_group != 1) return cudaErrorInvalidValue;
            switch (l.block_n) {
                case 64: return launch_tc_cfg<1, 64, kEpiPlain, KC, 2>(l);
                case 128: return launch_tc_cfg<1, 128, kEpiPlain, KC, 2>(l);
                default: return cudaErrorInvalidValue;
            }
        }
        return cudaErrorInvalidValue;
    }
    if (l.cta_group == 2) {
        switch (l.block_n) {
            case 256: return launch_tc_cfg<2, 256, kEpiPlain, KC>(l);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (l.block_n) {
        case 64: return launch_tc_cfg<1, 64, kEpiPlain, KC>(l);
        case 128: return launch_tc_cfg<1, 128, kEpiPlain, KC>(l);
        case 256: return launch_tc_cfg<1, 256, kEpiPlain, KC>(l);   // KC = 2: convolutions
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t GEMM103_CAT(launch_tc_, KERN_SUFFIX)(const TcLaunch& l) {
    if (l.esize != KERN_ES) return cudaErrorInvalidValue;
    if (l.kc == 1) return launch_tc_kc<1>(l);
    if (l.kc == 2) return launch_tc_kc<2>(l);
    return cudaErrorInvalidValue;
}

}  // namespace gemm103

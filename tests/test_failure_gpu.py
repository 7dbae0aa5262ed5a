"""Failure detection on the GPU without a fault: a bounded in-kernel wait that
nothing completes must come back as GEMM_ERR_DEVICE_TIMEOUT, and the handle
and the CUDA context must keep working afterwards."""
import time

import pytest
import torch

import gpu_cases as gc
import workloads

pytestmark = pytest.mark.gpu

LIMIT_NS = 200_000_000      # 0.2 s per wait


def _args(w, inp, A, B, C):
    return (w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(), inp.lda, B.data_ptr(),
            inp.ldb, w.beta, C.data_ptr(), inp.ldc, (w.ab_dtype, w.ab_dtype, w.c_dtype))


# 50 pair tiles of 256 x 256, fewer than the SM pairs: stream-K over CTA pairs
PAIR_SK = workloads.Workload("pair_sk_6272x512x4608", 6272, 512, 4608, "N", "T", workloads.DT_BF16,
                             workloads.DT_F32, 1.0, 0.0, "U", "U")


@pytest.mark.parametrize("name", ["square1024_f16_nt_f16out",       # single-CTA tiles
                                  "skinny_64x16384x8192_f16",       # stream-K, split tiles
                                  "linear_8192x4096x4096_bf16",     # CTA pairs
                                  "pair_sk"])                       # stream-K on CTA pairs
def test_timeout_is_reported_and_handle_recovers(orc, name):
    import mixed_precision_dense_sm_gb300 as lib
    w = PAIR_SK if name == "pair_sk" else workloads.WORKLOADS[name]
    if name == "pair_sk":
        lda, ldb, ldc = w.lds()
        st, plan = lib.gemm_plan_query("N", "T", w.M, w.N, w.K, 1.0, 256, lda, 256, ldb, 0.0, 256,
                                       ldc, (w.ab_dtype, w.ab_dtype, w.c_dtype),
                                       num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        assert st == 0 and plan["path_name"] == "tiled_2sm" and plan["sk_len"] > 0, plan
    inp = workloads.make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    C = torch.zeros((w.M, inp.ldc), dtype=workloads.TORCH_DTYPE[w.c_dtype], device="cuda")
    g = lib.Gemm()
    s = torch.cuda.current_stream().cuda_stream
    try:
        assert lib.gemm_debug_set(g.h, lib.GEMM_DEBUG_SKIP_FIRST_LOAD, LIMIT_NS) == 0
        t0 = time.time()
        assert lib.gemm_run(g.h, *_args(w, inp, A, B, C), s) == 0
        assert lib.gemm_sync(g.h, s) == 5                      # GEMM_ERR_DEVICE_TIMEOUT
        assert time.time() - t0 < 15.0
        assert lib.gemm_sync(g.h, s) == 0                      # reported once

        # a timeout recorded by one call is reported by the next gemm_run
        assert lib.gemm_run(g.h, *_args(w, inp, A, B, C), s) == 0
        torch.cuda.synchronize()
        assert lib.gemm_debug_set(g.h, 0, 0) == 0
        assert lib.gemm_run(g.h, *_args(w, inp, A, B, C), s) == 5
        torch.cuda.synchronize()

        # normal operation resumes on the same handle and context
        C.zero_()
        assert lib.gemm_run(g.h, *_args(w, inp, A, B, C), s) == 0
        assert lib.gemm_sync(g.h, s) == 0
        if w.M * w.N * w.K <= 2 ** 31:
            gc.check_full(orc, w, inp, C)
        else:
            gc.check_sampled(orc, w, inp, C, nsamp=1024)
    finally:
        lib.gemm_debug_set(g.h, 0, 0)
        g.close()

"""Host logic of the implicit-GEMM convolution (include/conv_sm103.h), no
GPU: output sizes, argument checks and the GEMM plan."""
import pytest

import mixed_precision_dense_sm_gb300 as lib
from workloads import DT_BF16, DT_F16, DT_F32

OK, INVALID, UNSUPPORTED = 0, 1, 2
F16 = (DT_F16, DT_F16, DT_F32)


def plan(N=2, H=8, W=8, C=64, K=64, R=3, S=3, pad=(1, 1), stride=(1, 1), dil=(1, 1), alpha=1.0,
         X=256, Wt=512, beta=0.0, Y=1 << 44, dt=F16, sms=152):
    return lib.conv2d_plan_query(N, H, W, C, K, R, S, pad, stride, dil, alpha, X, Wt, beta, Y, dt,
                                 num_sms=sms)


def test_exports():
    for name in ("conv2d_fprop", "conv2d_plan_query", "conv2d_output_dims"):
        assert name in lib.declared_symbols() and hasattr(lib.lib, name)


@pytest.mark.parametrize("geo", [(56, 56, 3, 3, (1, 1), (1, 1), (1, 1)),
                                 (7, 9, 3, 2, (0, 1), (2, 3), (2, 1)),
                                 (8, 9, 3, 3, (1, 1), (2, 2), (1, 1)),
                                 (3, 3, 5, 1, (0, 0), (1, 1), (1, 1)),
                                 (224, 224, 7, 7, (3, 3), (2, 2), (1, 1))])
def test_output_dims_match_the_oracle(orc, geo):
    H, W, R, S, pad, stride, dil = geo
    assert lib.conv2d_output_dims(H, W, R, S, pad, stride, dil) == \
        orc.conv2d_dims(H, W, R, S, pad[0], pad[1], stride[0], stride[1], dil[0], dil[1])


def test_plan_is_the_gemm_of_the_convolution():
    # k_blocks counts pipeline stages: 9 taps x ceil(C / 64) chunks of 64
    # channels, two chunks per stage when C is a multiple of 64
    st, p = plan(N=32, H=56, W=56, C=64, K=64)
    assert st == OK and p["k_blocks"] == 5 and p["block_k"] == 128
    assert p["tiles_m"] * 128 >= 32 * 56 * 56
    assert p["swap_ab"] == 0 and p["pack_a"] == 0 and p["pack_b"] == 0
    assert p["a_mn_major"] == 0 and p["b_mn_major"] == 0
    st, p = plan(N=16, H=64, W=64, C=256, K=256)
    assert st == OK and p["path_name"] == "tiled_2sm" and p["k_blocks"] == 9 * 4 // 2
    st, p = plan(N=2, H=12, W=10, C=72, K=40, R=5, S=5, pad=(2, 2))
    assert st == OK and p["k_blocks"] == 25 * 2                 # 72 channels: 2 blocks of 64
    assert p["block_k"] == 64                                   # one chunk per stage
    # few output pixels never swap (the im2col load fills the 128-row side);
    # a long reduction then runs stream-K
    st, p = plan(N=1, H=8, W=8, C=512, K=256)
    assert st == OK and p["swap_ab"] == 0 and p["sk_len"] > 0
    # empty output and alpha = 0 read nothing
    assert plan(N=0)[1]["path_name"] == "noop"
    assert plan(alpha=0.0, X=0, Wt=0, beta=1.0)[1]["path_name"] == "scale"


def test_argument_checks():
    for bad in [dict(C=0), dict(K=0), dict(R=0), dict(N=-1), dict(pad=(-1, 0)), dict(stride=(0, 1)),
                dict(dil=(1, 0)), dict(dt=(DT_F16, DT_BF16, DT_F32)), dict(dt=(DT_F32, DT_F32, DT_F32)),
                dict(dt=(DT_F16, DT_F16, 7)), dict(Y=0), dict(Y=2), dict(X=0)]:
        assert plan(**bad)[0] == INVALID, bad
    # limits of the im2col load
    for bad in [dict(C=12), dict(stride=(9, 1)), dict(pad=(129, 0)), dict(R=3, dil=(100, 1), H=300),
                dict(X=264), dict(Wt=520)]:
        assert plan(**bad)[0] == UNSUPPORTED, bad
    assert plan(C=8)[0] == OK and plan(stride=(8, 8))[0] == OK

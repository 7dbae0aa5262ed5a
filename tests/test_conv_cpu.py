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
    # im2col tiles (stride 2): k_blocks counts pipeline stages, 9 taps x
    # ceil(C / 64) chunks of 64 channels, two chunks per stage when C is a
    # multiple of 64
    st, p = plan(N=32, H=112, W=112, C=64, K=64, stride=(2, 2))
    assert st == OK and p["k_blocks"] == 5 and p["block_k"] == 128 and p["conv_rows"] == 0
    assert p["swap_ab"] == 0 and p["pack_a"] == 0 and p["pack_b"] == 0
    assert p["a_mn_major"] == 0 and p["b_mn_major"] == 0
    # halo units (stride 1): one step per filter column and channel block;
    # 32 images x 14 tiles of 4 output rows (4 x 56 <= 256)
    st, p = plan(N=32, H=56, W=56, C=64, K=64)
    assert st == OK and p["k_blocks"] == 3 and p["block_k"] == 64
    assert p["conv_rows"] == 4 and p["conv_pitch"] == 56 and p["tiles_m"] == 32 * 14
    assert p["block_m"] == 256 and p["stages"] >= 2
    st, p = plan(N=16, H=64, W=64, C=256, K=256)
    assert st == OK and p["path_name"] == "tiled_2sm" and p["k_blocks"] == 9 * 4 // 2
    st, p = plan(N=2, H=12, W=10, C=72, K=40, R=5, S=5, pad=(2, 2))
    assert st == OK and p["conv_pitch"] == 16 and p["k_blocks"] == 5 * 2   # 72 channels: 2 blocks
    st, p = plan(N=2, H=12, W=10, C=72, K=40, R=5, S=5, pad=(2, 2), stride=(1, 2))
    assert st == OK and p["k_blocks"] == 25 * 2 and p["block_k"] == 64     # one chunk per stage
    # few output pixels never swap (the im2col load fills the 128-row side);
    # a long reduction then runs stream-K
    st, p = plan(N=1, H=8, W=8, C=512, K=256)
    assert st == OK and p["swap_ab"] == 0 and p["sk_len"] > 0
    # empty output and alpha = 0 read nothing
    assert plan(N=0)[1]["path_name"] == "noop"
    assert plan(alpha=0.0, X=0, Wt=0, beta=1.0)[1]["path_name"] == "scale"


@pytest.mark.parametrize("H,W,stride,R,K,rows,pitch,halo", [
    (56, 56, 1, 3, 64, 4, 56, True), (28, 28, 1, 3, 128, 7, 32, True),
    (14, 14, 1, 3, 64, 14, 16, True), (9, 300, 1, 3, 64, 0, 0, False),
    (56, 56, 2, 3, 64, 0, 0, False), (64, 64, 1, 3, 256, 0, 0, False),
    (17, 17, 1, 1, 96, 9, 24, True), (40, 50, 1, 5, 64, 4, 56, True),
    (8, 250, 1, 3, 64, 1, 250, False)])
def test_whole_row_tiles(H, W, stride, R, K, rows, pitch, halo):
    """Stride-1 convolutions on 256-row single-CTA tiles (at most 128 output
    channels) tile each image by whole output rows at a pitch of A rows per
    output row, T pitch <= 256, the rows split evenly: tiles per image =
    ceil(P / floor(256 / pitch)), T = ceil(P / that).  Halo units (pitch = Q
    rounded up to 8) take one step per filter column and channel block; where
    their stages do not fit two to shared memory (250-pixel rows) each tap
    loads its own box (pitch = Q, one step per tap).  Strided layers, rows
    wider than 256 pixels and CTA-pair tiles keep the im2col tiles."""
    pad = (R // 2, R // 2)
    st, p = plan(N=3, H=H, W=W, C=64, K=K, R=R, S=R, pad=pad, stride=(stride, stride))
    assert st == OK and p["conv_rows"] == rows and p["conv_pitch"] == pitch, p
    if rows:
        P = (H + 2 * pad[0] - R) // stride + 1
        Q = (W + 2 * pad[1] - R) // stride + 1
        tpi = p["tiles_m"] // 3
        assert p["tiles_m"] == 3 * tpi and tpi == -(-P // (256 // pitch))
        assert rows == -(-P // tpi) and rows * pitch <= 256 and (tpi - 1) * rows < P
        assert p["block_m"] == 256 and p["path_name"] == "tiled_1sm" and p["sk_len"] == 0
        assert pitch == (-(-Q // 8) * 8 if halo else Q)
        assert p["k_blocks"] == (R if halo else -(-R * R // 2)), p


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


def test_whole_row_plan_invariants_on_random_layers():
    """Seeded random stride-1 and strided layers: every whole-row plan keeps
    its tile inside 256 rows at its pitch, covers each image's output rows
    exactly once with the rows split evenly, and is a halo plan (pitch Q
    rounded up to 8, k_blocks = S ceil(C / 64), a box of at most 256 rows)
    or a box-per-tap plan (pitch Q); layers without whole-row tiles are
    strided, have rows wider than 256 pixels, or run other tiles."""
    import random
    rng = random.Random(20261202)
    seen_halo = seen_tap = seen_none = 0
    for _ in range(400):
        R = rng.choice([1, 3, 5, 7])
        S = rng.choice([1, 3, 5])
        dil = (rng.choice([1, 1, 2]), rng.choice([1, 1, 2]))
        stride = (1, 1) if rng.random() < 0.8 else (rng.choice([1, 2]), 2)
        H = rng.randint((R - 1) * dil[0] + 1, 80)
        W = rng.choice([rng.randint((S - 1) * dil[1] + 1, 64), rng.randint(200, 300)])
        C = 8 * rng.randint(1, 40)
        K = rng.choice([16, 40, 64, 96, 128, 256])
        N = rng.randint(1, 6)
        pad = (rng.randint(0, R // 2 * dil[0]), rng.randint(0, S // 2 * dil[1]))
        st, p = plan(N=N, H=H, W=W, C=C, K=K, R=R, S=S, pad=pad, stride=stride, dil=dil)
        if st != OK or p["path_name"] in ("noop", "scale"):
            continue
        P = (H + 2 * pad[0] - dil[0] * (R - 1) - 1) // stride[0] + 1
        Q = (W + 2 * pad[1] - dil[1] * (S - 1) - 1) // stride[1] + 1
        rows, pitch = p["conv_rows"], p["conv_pitch"]
        if rows == 0:
            assert pitch == 0
            assert stride != (1, 1) or Q > 256 or p["block_m"] != 256 or \
                p["path_name"] != "tiled_1sm", (N, H, W, C, K, R, S, pad, stride, dil, p)
            seen_none += 1
            continue
        assert stride == (1, 1) and p["path_name"] == "tiled_1sm" and p["block_m"] == 256
        assert p["block_n"] <= 128 and rows * pitch <= 256 and pitch in (Q, -(-Q // 8) * 8)
        tpi = p["tiles_m"] // N
        assert p["tiles_m"] == N * tpi and (tpi - 1) * rows < P <= tpi * rows
        assert rows == -(-P // tpi)
        cb = -(-C // 64)
        kc = 2 if C % 64 == 0 else 1
        tap_blocks = -(-R * S * cb // kc)
        if pitch != Q or (p["k_blocks"] != tap_blocks and p["k_blocks"] == S * cb):
            # halo units: one step per filter column and channel block
            assert pitch == -(-Q // 8) * 8 and p["k_blocks"] == S * cb
            assert rows + (R - 1) * dil[0] <= 256 and p["stages"] >= 2
            seen_halo += 1
        else:
            # a box per tap (or a halo plan that no count tells apart)
            assert p["k_blocks"] in (tap_blocks, S * cb)
            seen_tap += 1
    assert seen_halo > 50 and seen_none > 20

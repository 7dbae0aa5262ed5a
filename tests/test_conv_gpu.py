"""GPU parity of the implicit-GEMM convolution (CATLASS page, section 5.1):
conv2d_fprop through the C ABI against the CPU oracle -- padding, stride,
dilation, channel counts that do not fill a 64-channel block, every output
type, alpha / beta, the fused epilogue, CTA pairs and stream-K."""
import numpy as np
import pytest
import torch

import checks
import workloads
from workloads import DT_BF16, DT_F16, DT_F32, TORCH_DTYPE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import mixed_precision_dense_sm_gb300 as lib
    h = lib.Gemm()
    yield h
    h.close()


def make(N, H, W, C, K, R, S, dt, integer, seed):
    gen = torch.Generator().manual_seed(seed)
    if integer:
        x = torch.randint(-3, 4, (N, H, W, C), generator=gen).float()
        w = torch.randint(-3, 4, (K, R, S, C), generator=gen).float()
    else:
        x = torch.randn((N, H, W, C), generator=gen)
        w = torch.randn((K, R, S, C), generator=gen) * 0.1
    return x.to(TORCH_DTYPE[dt]), w.to(TORCH_DTYPE[dt])


def run_and_check(g, orc, geo, dt=DT_BF16, ydt=DT_F32, alpha=1.0, beta=0.0, integer=True,
                  seed=0, bias=False, act=0, sample=None):
    import mixed_precision_dense_sm_gb300 as lib
    N, H, W, C, K, R, S, pad, stride, dil = geo
    P, Q = lib.conv2d_output_dims(H, W, R, S, pad, stride, dil)
    M = N * P * Q
    x, w = make(N, H, W, C, K, R, S, dt, integer, seed)
    gen = torch.Generator().manual_seed(seed + 7)
    yin = (torch.randint(-3, 4, (M, K), generator=gen).float() if integer
           else torch.randn((M, K), generator=gen)).to(TORCH_DTYPE[ydt])
    bvec = (torch.randint(-3, 4, (K,), generator=gen).float() if integer
            else torch.randn((K,), generator=gen) * 0.1).to(torch.float32) if bias else None
    X, Wd = x.cuda(), w.cuda()
    Y = yin.clone().cuda() if beta != 0 else torch.full((M, K), float("nan"), dtype=TORCH_DTYPE[ydt],
                                                         device="cuda")
    B = bvec.cuda() if bias else None
    st = lib.conv2d_fprop(g.h, N, H, W, C, K, R, S, pad, stride, dil, alpha, X.data_ptr(),
                          Wd.data_ptr(), beta, Y.data_ptr(), (dt, dt, ydt),
                          B.data_ptr() if bias else 0, DT_F32, act,
                          torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.gemm_status_string(st)
    g.sync()
    xc, wc = workloads.as_codes(x), workloads.as_codes(w)
    yc = workloads.as_codes(yin) if beta != 0 else None
    args = (N, H, W, C, K, R, S, pad[0], pad[1], stride[0], stride[1], dil[0], dil[1], alpha, xc, wc,
            beta, yc, dt, ydt)
    rows = np.arange(M) if sample is None else sample(M)
    if sample is None:
        Rr, Sr = orc.conv2d(*args)
    else:
        Rr, Sr = orc.conv2d_sampled(*args, rows)
    if bias or act:
        bv = bvec.double().numpy() if bias else np.zeros(K)
        Rr = np.vectorize(lambda v: orc.activation(act, v))(Rr + bv) if act else Rr + bv
        Sr = Sr + np.abs(bv)
    got = Y.cpu()[torch.as_tensor(rows)]
    vals = got.double().numpy()
    codes = None if ydt == DT_F32 else got.contiguous().view(torch.int16).numpy().view(np.uint16)
    ocodes = None if ydt == DT_F32 else orc.round_output(Rr, ydt)
    cin = yin.double().numpy()[rows] if beta != 0 else None
    if integer and not act:
        want = orc.round_output(Rr, DT_F32).astype(np.float64) if ydt == DT_F32 else None
        bad = (vals != want) if ydt == DT_F32 else (codes != ocodes)
        assert not bad.any(), f"{geo}: {int(bad.sum())} of {bad.size} differ from the exact result"
        return {"exact": True, "n": int(bad.size)}
    if act:
        stats, bad = checks.compare_epilogue(vals, codes, Rr, Sr, cin, None, alpha, beta, ydt, ocodes)
    else:
        stats, bad = checks.compare(vals, codes, Rr, Sr, cin, alpha, beta, ydt, ocodes)
    if stats["fail"]:
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{geo}: {stats}; first bad ({rows[i]}, {j}) gpu={vals[i, j]!r} "
                             f"oracle={Rr[i, j]!r}")
    return stats


GEOS = [
    # N, H, W, C, K, R, S, pad, stride, dilation
    (1, 5, 6, 8, 16, 3, 3, (1, 1), (1, 1), (1, 1)),
    (2, 9, 7, 16, 24, 3, 2, (0, 1), (2, 3), (2, 1)),
    (1, 8, 8, 64, 64, 1, 1, (0, 0), (1, 1), (1, 1)),
    (2, 12, 10, 72, 40, 5, 5, (2, 2), (1, 1), (1, 1)),
    (1, 16, 16, 128, 130, 3, 3, (1, 1), (2, 2), (1, 1)),
    (3, 7, 7, 8, 8, 7, 7, (3, 3), (1, 1), (1, 1)),
    (1, 31, 29, 32, 64, 3, 3, (1, 1), (2, 1), (1, 2)),
    (4, 20, 20, 16, 32, 3, 3, (1, 1), (1, 1), (1, 1)),
    (2, 11, 13, 200, 96, 2, 3, (0, 2), (3, 2), (2, 3)),
    (1, 6, 6, 8, 8, 3, 3, (5, 0), (1, 1), (1, 1)),        # windows entirely in the padding
]


@pytest.mark.parametrize("geo", GEOS, ids=[f"g{i}" for i in range(len(GEOS))])
def test_geometries_integer_exact(g, orc, geo):
    """Integer inputs keep every FP32 partial sum exact: the result must be
    bit-identical to the oracle's, whatever the padding, stride and dilation."""
    run_and_check(g, orc, geo, dt=(DT_BF16, DT_F16)[hash(geo) % 2], ydt=DT_F32, seed=sum(geo[:7]))


WHOLE_ROWS = [
    # N, H, W, C, K, R, S, pad, stride, dilation; halo units?
    ((3, 23, 21, 64, 64, 3, 3, (1, 1), (1, 1), (1, 1)), True),    # 8 rows per tile, the last 7
    ((2, 30, 40, 24, 40, 3, 3, (2, 2), (1, 1), (2, 2)), True),    # dilation 2, 24 channels
    ((2, 9, 130, 64, 128, 3, 5, (1, 2), (1, 1), (1, 1)), False),  # 130-pixel rows: a box per tap
    ((1, 33, 33, 128, 96, 1, 1, (0, 0), (1, 1), (1, 1)), True),   # 1 x 1: 6 rows, the last 3
    ((2, 20, 19, 16, 32, 7, 7, (3, 3), (1, 1), (1, 1)), True),    # 7 x 7: 16-row halo boxes
    ((2, 15, 26, 40, 48, 3, 3, (2, 1), (1, 1), (2, 1)), True),    # dilation (2, 1), pitch 32
    ((2, 22, 9, 136, 72, 3, 3, (0, 1), (1, 1), (1, 1)), True),    # 3 channel blocks, no row pad
]


@pytest.mark.parametrize("case", WHOLE_ROWS, ids=[f"r{i}" for i in range(len(WHOLE_ROWS))])
def test_whole_row_tiles(g, orc, case):
    """Stride-1 layers with at most 128 output channels run whole-row tiles:
    halo units (one tiled box of the input per filter column and channel
    block, the column's taps read at row offsets of it, rows at a pitch of Q
    rounded up to 8) or, where those stages do not fit, one box per tap
    (T output rows x Q pixels); zeros outside the image, rows past the
    image's last row and pitch columns past Q masked.  Integer inputs
    bit-exact, then random inputs with a 16-bit output."""
    import mixed_precision_dense_sm_gb300 as lib
    geo, halo = case
    st, p = lib.conv2d_plan_query(*geo, 1.0, 256, 256, 0.0, 1 << 44, (DT_BF16, DT_BF16, DT_F32),
                                  num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0 and p["conv_rows"] > 0, p
    C, S = geo[3], geo[6]
    assert (p["k_blocks"] == S * -(-C // 64)) == halo, p
    run_and_check(g, orc, geo, dt=DT_BF16, ydt=DT_F32, seed=sum(geo[:7]))
    run_and_check(g, orc, geo, dt=DT_F16, ydt=DT_BF16, integer=False, beta=0.5, seed=3)


@pytest.mark.parametrize("ydt", [DT_F32, DT_F16, DT_BF16])
def test_random_every_output_type(g, orc, ydt):
    for i, geo in enumerate(GEOS[:8]):
        dt = (DT_F16, DT_BF16)[i % 2]
        stats = run_and_check(g, orc, geo, dt=dt, ydt=ydt, alpha=(1.0, 0.5)[i % 2],
                              beta=(0.0, -1.0)[(i // 2) % 2], integer=False, seed=i)
        print(geo, stats)


def test_fused_epilogue(g, orc):
    """Bias per output channel and each activation, on the convolution."""
    for act in (0, 1, 2, 3):
        run_and_check(g, orc, GEOS[3], dt=DT_BF16, ydt=DT_BF16, bias=True, act=act, integer=False,
                      seed=act)


def test_cta_pairs_and_stream_k(g, orc):
    """A layer large enough for 256 x 256 CTA-pair tiles, and one with few
    output pixels and a long reduction (stream-K), sampled outputs."""
    import mixed_precision_dense_sm_gb300 as lib
    big = (16, 32, 32, 64, 512, 3, 3, (1, 1), (1, 1), (1, 1))
    st, p = lib.conv2d_plan_query(*big, 1.0, 256, 256, 0.0, 1 << 44, (DT_BF16, DT_BF16, DT_BF16),
                                  num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0 and p["path_name"] == "tiled_2sm", p
    sample = lambda M: np.unique(np.concatenate([np.arange(0, M, 97), [M - 1, 1, 2]]))
    run_and_check(g, orc, big, dt=DT_BF16, ydt=DT_BF16, integer=True, sample=sample)
    run_and_check(g, orc, big, dt=DT_F16, ydt=DT_F32, integer=False, beta=1.0, sample=sample)
    long_k = (1, 8, 8, 512, 256, 3, 3, (1, 1), (1, 1), (1, 1))
    st, p = lib.conv2d_plan_query(*long_k, 1.0, 256, 256, 0.0, 1 << 44, (DT_BF16, DT_BF16, DT_F32),
                                  num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0 and p["sk_len"] > 0, p
    run_and_check(g, orc, long_k, dt=DT_BF16, ydt=DT_F32, integer=True)
    run_and_check(g, orc, long_k, dt=DT_BF16, ydt=DT_BF16, integer=False, seed=3)


def test_pair_stream_k_full_layer(g, orc):
    """The 32 x 14 x 14, C = K = 512 layer: 50 CTA-pair tiles, fewer than the
    SM pairs, with two K chunks per stage in three stages and stream-K over
    36 stages per tile; sampled pixels (every 37th and the last) against the
    oracle, both input types."""
    import mixed_precision_dense_sm_gb300 as lib
    geo = (32, 14, 14, 512, 512, 3, 3, (1, 1), (1, 1), (1, 1))
    st, p = lib.conv2d_plan_query(*geo, 1.0, 256, 256, 0.0, 1 << 44, (DT_BF16, DT_BF16, DT_BF16),
                                  num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0 and (p["path_name"], p["block_n"], p["block_k"], p["stages"]) == \
        ("tiled_2sm", 256, 128, 3) and p["sk_len"] > 0, p
    sample = lambda M: np.unique(np.concatenate([np.arange(0, M, 37), [M - 1, 1, 2]]))
    run_and_check(g, orc, geo, dt=DT_BF16, ydt=DT_BF16, integer=True, sample=sample)
    run_and_check(g, orc, geo, dt=DT_F16, ydt=DT_F32, integer=False, beta=1.0, sample=sample)


def test_single_cta_wide_tiles_two_chunks(g, orc):
    """196 output pixels by 19456 filters, C = 64: 152 single-CTA 256-wide
    tiles with two K chunks per stage in two stages (the operands are re-read
    from L2); sampled pixels against the oracle."""
    import mixed_precision_dense_sm_gb300 as lib
    geo = (1, 14, 14, 64, 19456, 3, 3, (1, 1), (1, 1), (1, 1))
    st, p = lib.conv2d_plan_query(*geo, 1.0, 256, 256, 0.0, 1 << 44, (DT_BF16, DT_BF16, DT_BF16),
                                  num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0 and (p["path_name"], p["block_n"], p["block_k"], p["stages"]) == \
        ("tiled_1sm", 256, 128, 2), p
    sample = lambda M: np.unique(np.concatenate([np.arange(0, M, 13), [M - 1, 1, 2]]))
    run_and_check(g, orc, geo, dt=DT_BF16, ydt=DT_BF16, integer=True, sample=sample)


@pytest.mark.parametrize("name", list(workloads.CONV_WORKLOADS))
def test_conv_workloads_sampled(g, orc, name):
    """The named convolution layers at full size, with the benchmark's seeded
    inputs and in the launch configuration it times (halo units for the
    64- and 128-channel layers, CTA pairs and stream-K for the others):
    sampled output pixels -- the first and last of every image and a spread
    between -- against the oracle, every output channel."""
    import mixed_precision_dense_sm_gb300 as lib
    w = workloads.CONV_WORKLOADS[name]
    x, wt = workloads.make_conv_inputs(w)
    P, Q = w.out_hw()
    M = w.N * P * Q
    X, Wd = x.cuda(), wt.cuda()
    Y = torch.full((M, w.K), float("nan"), dtype=TORCH_DTYPE[w.y_dtype], device="cuda")
    st = lib.conv2d_fprop(g.h, w.N, w.H, w.W, w.C, w.K, w.R, w.S, w.pad, w.stride, w.dil, 1.0,
                          X.data_ptr(), Wd.data_ptr(), 0.0, Y.data_ptr(),
                          (w.x_dtype, w.x_dtype, w.y_dtype), 0, DT_F32, 0,
                          torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.gemm_status_string(st)
    g.sync()
    per = P * Q
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 700)), np.arange(0, M, per),
                                     np.arange(per - 1, M, per), [1, Q, Q + 1]]))
    xc, wc = workloads.as_codes(x), workloads.as_codes(wt)
    Rr, Sr = orc.conv2d_sampled(w.N, w.H, w.W, w.C, w.K, w.R, w.S, w.pad[0], w.pad[1], w.stride[0],
                                w.stride[1], w.dil[0], w.dil[1], 1.0, xc, wc, 0.0, None,
                                w.x_dtype, w.y_dtype, rows)
    got = Y.cpu()[torch.as_tensor(rows)]
    vals = got.double().numpy()
    codes = None if w.y_dtype == DT_F32 else got.contiguous().view(torch.int16).numpy().view(np.uint16)
    ocodes = None if w.y_dtype == DT_F32 else orc.round_output(Rr, w.y_dtype)
    stats, bad = checks.compare(vals, codes, Rr, Sr, None, 1.0, 0.0, w.y_dtype, ocodes)
    if stats["fail"]:
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{name}: {stats}; first bad ({rows[i]}, {j}) gpu={vals[i, j]!r} "
                             f"oracle={Rr[i, j]!r}")
    print(name, len(rows), "pixels", stats)


def test_errors_enqueue_nothing(g):
    import mixed_precision_dense_sm_gb300 as lib
    Y = torch.full((64, 16), 5.0, device="cuda")
    X = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    geo = (1, 8, 8, 8, 16, 3, 3, (1, 1), (1, 1), (1, 1))
    assert lib.conv2d_fprop(g.h, *geo[:7], (1, 1), (1, 1), (1, 1), 1.0, X.data_ptr(), X.data_ptr(),
                            0.0, Y.data_ptr(), (DT_BF16, DT_F16, DT_F32)) == 1
    assert lib.conv2d_fprop(g.h, 1, 8, 8, 12, 16, 3, 3, (1, 1), (1, 1), (1, 1), 1.0, X.data_ptr(),
                            X.data_ptr(), 0.0, Y.data_ptr(), (DT_BF16, DT_BF16, DT_F32)) == 2
    assert lib.conv2d_fprop(g.h, 1, 8, 8, 8, 16, 3, 3, (1, 1), (1, 1), (1, 1), 1.0,
                            X.data_ptr() + 2, X.data_ptr(), 0.0, Y.data_ptr(),
                            (DT_BF16, DT_BF16, DT_F32)) == 2
    g.sync()
    assert torch.all(Y == 5.0)

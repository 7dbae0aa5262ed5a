"""GPU parity of the row softmax (SGEMM tutorial page, section 2): the CUDA
path through the C ABI against the CPU oracle, on every work split (warp,
CTA, cluster, two-pass), every input/output type, aligned and unaligned rows
and the special values."""
import itertools

import numpy as np
import pytest
import torch

import checks
import workloads
from workloads import DT_BF16, DT_F16, DT_F32, TORCH_DTYPE, SoftmaxWorkload

pytestmark = pytest.mark.gpu

CANARY = 1234.5


@pytest.fixture(scope="module")
def lib():
    import mixed_precision_dense_sm_gb300 as m
    return m


def stored(values: torch.Tensor, ld: int, dt: int) -> torch.Tensor:
    rows, cols = values.shape
    buf = torch.full((rows, max(ld, 1)), float("nan"), dtype=TORCH_DTYPE[dt])
    buf[:, :cols] = values.to(TORCH_DTYPE[dt])
    return buf


def to_device(t: torch.Tensor, misalign: bool) -> torch.Tensor:
    if not misalign:
        return t.cuda()
    rows, ld = t.shape
    flat = torch.empty(rows * ld + 8, dtype=t.dtype, device="cuda")
    view = flat[1:1 + rows * ld].view(rows, ld)
    view.copy_(t)
    return view


def run(lib, Xs: torch.Tensor, cols: int, y_dt: int, ldy=None, misalign=False, inplace=False):
    """Xs: stored CPU rows x ldx tensor.  Returns the device Y (stored)."""
    rows, ldx = Xs.shape
    X = to_device(Xs, misalign)
    if inplace:
        Y, ldy = X, ldx
    else:
        ldy = ldy or max(cols, 1)
        Yh = torch.full((rows, ldy), CANARY, dtype=TORCH_DTYPE[y_dt])
        Y = to_device(Yh, misalign)
    s = torch.cuda.current_stream().cuda_stream
    st = lib.softmax_rows(rows, cols, X.data_ptr(), ldx, lib.dtype_code(X.dtype), Y.data_ptr(),
                          ldy, y_dt, s)
    assert st == 0, lib.gemm_status_string(st)
    torch.cuda.synchronize()
    return Y


def check(orc, Xs: torch.Tensor, cols: int, x_dt: int, y_dt: int, Y: torch.Tensor, row_ids=None,
          canary=True):
    rows, ldx = Xs.shape
    R = orc.softmax(workloads.as_codes(Xs), rows, cols, ldx, x_dt, row_ids=row_ids)
    ids = np.arange(rows) if row_ids is None else np.asarray(row_ids)
    Xv = Xs[ids][:, :cols].to(torch.float64).numpy()
    Yc = Y[torch.as_tensor(ids, device=Y.device)][:, :cols].cpu()
    vals = Yc.to(torch.float64).numpy()
    codes = ocodes = None
    if y_dt != DT_F32:
        codes = Yc.contiguous().view(torch.int16).numpy().view(np.uint16)
        ocodes = orc.round_output(R, y_dt)
    stats, bad = checks.compare_softmax(vals, codes, R, Xv, y_dt, ocodes)
    if stats["fail"]:
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{stats}; first bad row {ids[i]} col {j}: gpu={vals[i, j]!r} "
                             f"oracle={R[i, j]!r} x={Xv[i, j]!r}")
    if canary and Y.shape[1] > cols:
        pad = Y[:, cols:].float().cpu()
        want = torch.tensor(CANARY).to(Y.dtype).float()    # the canary as stored in Y's type
        assert torch.all(pad == want), "Y padding was written"
    return stats


COLS = [1, 2, 7, 31, 32, 33, 100, 1000, 1024, 1025, 2049, 4096, 8192, 8193, 12345, 16384,
        16385, 16392, 32768, 40000, 65536, 100000, 131072, 131073, 300001]


@pytest.mark.parametrize("cols", COLS)
def test_every_work_split(lib, orc, cols):
    """Ragged and exact row lengths on each side of every split boundary
    (warp 1024, CTA 8192 / 16384, two passes above 16384 -- the rows
    streamed twice through shared memory in 32 KB chunks, by one CTA or,
    above about 110000, by a cluster of 2-4), 16-byte aligned rows, FP32 in
    and out, 4 N(0,1) logits."""
    rows = 5 if cols > 20000 else 37
    g = torch.Generator().manual_seed(cols)
    x = torch.randn((rows, cols), generator=g) * 4.0
    Xs = stored(x, cols + (-cols) % 8, DT_F32)
    Y = run(lib, Xs, cols, DT_F32, ldy=cols + (-cols) % 8 + 8)
    check(orc, Xs, cols, DT_F32, DT_F32, Y)


@pytest.mark.parametrize("cols", [100, 5000, 40000, 200000])
def test_every_type_pair(lib, orc, cols):
    """All nine input/output type pairs on each work split."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn((6, cols), generator=g) * 3.0
    for xdt, ydt in itertools.product((DT_F32, DT_F16, DT_BF16), repeat=2):
        Xs = stored(x, cols + 8, xdt)
        Y = run(lib, Xs, cols, ydt, ldy=cols + 16)
        check(orc, Xs, cols, xdt, ydt, Y)


@pytest.mark.parametrize("cols,gw,unit", [(1024, 8, 8), (1001, 8, 8), (2048, 8, 8), (1536, 8, 8),
                                          (4096, 4, 1), (6001, 8, 1), (8192, 8, 1), (16000, 16, 1),
                                          (16384, 16, 1), (20000, 16, 1), (32768, 16, 1)])
def test_staged_16bit_splits(lib, orc, cols, gw, unit):
    """16-bit rows in the staged kernel: a warp per row up to 2048 elements
    (64 per lane), else groups of 4-16 warps that merge their warps' (max,
    sum) pairs;
    whole rows, rows whose vectors do not fill every thread and rows with a
    tail past the last 16-byte vector; FP16 and BF16 inputs with 16-bit and
    FP32 outputs; fully and half masked rows; more rows than slots."""
    rows = 300 if cols <= 8192 else 80
    ld = cols + (-cols) % 8
    st, p = lib.softmax_plan_query(rows, cols, 256, ld, DT_BF16, 1 << 44, ld, DT_BF16)
    assert st == 0 and p["depth"] > 0 and (p["group_warps"], p["unit_rows"]) == (gw, unit), p
    g = torch.Generator().manual_seed(cols + 3)
    x = torch.randn((rows, cols), generator=g) * 3.0
    x[1, :] = float("-inf")
    x[2, cols // 2:] = float("-inf")
    x[3, :cols // 3] = float("-inf")
    for xdt, ydt in [(DT_BF16, DT_BF16), (DT_F16, DT_F32), (DT_BF16, DT_F16)]:
        Xs = stored(x, ld, xdt)
        Y = run(lib, Xs, cols, ydt, ldy=ld)
        check(orc, Xs, cols, xdt, ydt, Y, canary=False)


@pytest.mark.parametrize("cols", [77, 1000, 3001, 9000, 20001, 140001])
def test_unaligned_rows(lib, orc, cols):
    """Row pitches that are not a multiple of 16 bytes and base addresses one
    element off: the element-by-element path of every split."""
    g = torch.Generator().manual_seed(cols + 1)
    x = torch.randn((9, cols), generator=g)
    for xdt, ydt in [(DT_F32, DT_F32), (DT_BF16, DT_F16), (DT_F16, DT_F32)]:
        Xs = stored(x, cols + 3, xdt)
        Y = run(lib, Xs, cols, ydt, ldy=cols + 5, misalign=True)
        check(orc, Xs, cols, xdt, ydt, Y)


@pytest.mark.parametrize("cols", [64, 3000, 24000, 150000])
def test_special_values(lib, orc, cols):
    """NaN or +inf in a row (NaN row), a fully masked row (0/0: NaN), single
    masked entries (exactly 0), a causal mask, and logits far beyond exp's
    range (only the max shift reaches them)."""
    g = torch.Generator().manual_seed(11)
    x = torch.randn((10, cols), generator=g)
    x[0, cols // 3] = float("nan")
    x[1, cols - 1] = float("inf")
    x[2, :] = float("-inf")
    x[3, ::5] = float("-inf")
    x[4, :] = x[4, :] * 1e4                          # FP32: exp far out of range
    keep = torch.arange(cols) <= (cols // 2)
    x[5, :] = torch.where(keep, x[5, :], torch.tensor(float("-inf")))
    x[6, 1:] = float("-inf")                         # one live entry
    x[7, :] = 0.0                                    # uniform
    x[8, :] = -3.0e4                                 # uniform, very negative
    for xdt, ydt in [(DT_F32, DT_F32), (DT_F16, DT_F16), (DT_BF16, DT_F32)]:
        xs = x.clone()
        if xdt == DT_F16:
            xs[4, :] = xs[4, :].clamp(-6e4, 6e4)
        Xs = stored(xs, cols + 8, xdt)
        Y = run(lib, Xs, cols, ydt, ldy=cols + 8)
        check(orc, Xs, cols, xdt, ydt, Y)
        yv = Y[:, :cols].float().cpu()
        assert torch.isnan(yv[0]).all() and torch.isnan(yv[1]).all() and torch.isnan(yv[2]).all()
        assert (yv[3, ::5] == 0).all() and (yv[6, 1:] == 0).all() and yv[6, 0] == 1.0


@pytest.mark.parametrize("cols", [1024, 8192, 16384, 65536, 262144])
def test_dominant_entry_everywhere(lib, orc, cols):
    """A row whose mass sits on one entry, placed at the first and last
    element and on each side of every vector, chunk and slice boundary: an
    element that is skipped or read twice changes the result at O(1)."""
    st, p = lib.softmax_plan_query(1, cols, 256, cols, DT_F32, 1 << 44, cols, DT_F32)
    assert st == 0
    marks = {0, cols - 1, cols // 2}
    for b in range(0, cols, 8 * max(1, cols // 64)):
        marks |= {b, b - 1, b + 7}
    for c in range(p["cluster"]):
        marks |= {c * p["slice"] - 1, c * p["slice"]}
    for ch in range(0, p["slice"], p["threads"] * 32):
        marks |= {ch - 1, ch}
    marks = sorted(m for m in marks if 0 <= m < cols)[:256]
    g = torch.Generator().manual_seed(3)
    x = torch.randn((len(marks), cols), generator=g)
    for r, m in enumerate(marks):
        x[r, m] = 40.0
    Xs = stored(x, cols, DT_F32)
    Y = run(lib, Xs, cols, DT_F32)
    check(orc, Xs, cols, DT_F32, DT_F32, Y)
    top = Y.argmax(dim=1).cpu()
    assert (top == torch.tensor(marks)).all()


def test_in_place_and_deterministic(lib, orc):
    """Y = X in place and three runs bitwise equal, in every split: warp
    rows, a staged CTA row, long rows on one CTA and (400000 elements) long
    rows on a cluster of 2."""
    for cols in (1000, 10000, 100000, 200000, 400000):
        g = torch.Generator().manual_seed(cols)
        Xs = stored(torch.randn((7, cols), generator=g), cols, DT_BF16)
        Y = run(lib, Xs, cols, DT_BF16, inplace=True)
        check(orc, Xs, cols, DT_BF16, DT_BF16, Y, canary=False)
        outs = [run(lib, Xs, cols, DT_BF16).cpu() for _ in range(3)]
        for o in outs[1:]:
            assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_many_rows_persistent(lib, orc):
    """More rows than resident row groups, in every split."""
    for rows, cols in [(20000, 64), (3000, 3000), (700, 20000), (40, 140000)]:
        g = torch.Generator().manual_seed(rows)
        Xs = stored(torch.randn((rows, cols), generator=g), cols, DT_F32)
        Y = run(lib, Xs, cols, DT_F32)
        ids = np.unique(np.concatenate([np.arange(0, rows, max(1, rows // 97)), [rows - 1]]))
        check(orc, Xs, cols, DT_F32, DT_F32, Y, row_ids=ids)


@pytest.mark.parametrize("name", list(workloads.SOFTMAX_WORKLOADS))
def test_workloads_sampled(lib, orc, name):
    """The named softmax workloads at full size, in the launch configuration
    the benchmark times; sampled rows (first, last and spread)."""
    w = workloads.SOFTMAX_WORKLOADS[name]
    Xs = workloads.make_softmax_input(w)
    ldx, ldy = w.lds()
    X = Xs.cuda()
    Y = torch.empty((w.rows, ldy), dtype=TORCH_DTYPE[w.y_dtype], device="cuda")
    st = lib.softmax_rows(w.rows, w.cols, X.data_ptr(), ldx, w.x_dtype, Y.data_ptr(), ldy,
                          w.y_dtype, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    n = min(w.rows, 48)
    ids = np.unique(np.concatenate([np.linspace(0, w.rows - 1, n).astype(np.int64), [1, 2]]))
    ids = ids[ids < w.rows]
    stats = check(orc, Xs, w.cols, w.x_dtype, w.y_dtype, Y, row_ids=ids, canary=False)
    print(name, stats)


def test_empty_and_errors(lib):
    s = torch.cuda.current_stream().cuda_stream
    Y = torch.full((4, 4), 7.0, device="cuda")
    assert lib.softmax_rows(0, 4, 0, 4, DT_F32, Y.data_ptr(), 4, DT_F32, s) == 0
    assert lib.softmax_rows(4, 0, 0, 4, DT_F32, Y.data_ptr(), 4, DT_F32, s) == 0
    assert lib.softmax_rows(4, 4, Y.data_ptr(), 3, DT_F32, Y.data_ptr(), 4, DT_F32, s) == 1
    assert lib.softmax_rows(4, 4, Y.data_ptr() + 2, 4, DT_F32, Y.data_ptr(), 4, DT_F32, s) == 1
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)


@pytest.mark.parametrize("cols", [1024, 4096, 16384, 65536, 262144])
def test_timeout_reported_without_fault(lib, orc, cols):
    """The failure path of the staged kernels, without a GPU fault: the test
    hook arms the first row slot of the first pipeline without issuing its
    copy, so that bounded wait runs out (limit 0.2 s).  softmax_sync reports
    GEMM_ERR_DEVICE_TIMEOUT once; the next call on the same device is
    correct.  1024 FP32 columns run a warp per row, 4096 a group of 8 warps
    per row, 16384 a group of 16 warps (every compute warp) per row, 65536
    the long-row kernel (the row streamed twice in chunks), 262144 that
    kernel with each row split over a cluster of 4 CTAs (the failing CTA
    keeps exchanging with its peers, so none waits for it unbounded)."""
    g = torch.Generator().manual_seed(5)
    Xs = stored(torch.randn((64, cols), generator=g), cols, DT_F32)
    st, p = lib.softmax_plan_query(64, cols, 256, cols, DT_F32, 1 << 44, cols, DT_F32)
    assert st == 0 and p["depth"] > 0
    s = torch.cuda.current_stream().cuda_stream
    assert lib.softmax_sync(s) == 0
    X = Xs.cuda()
    Y = torch.empty_like(X)
    assert lib.softmax_debug_set(lib.SOFTMAX_DEBUG_SKIP_FIRST_LOAD, 200_000_000) == 0
    try:
        assert lib.softmax_rows(64, cols, X.data_ptr(), cols, DT_F32, Y.data_ptr(), cols,
                                DT_F32, s) == 0
        assert lib.softmax_sync(s) == 5
    finally:
        assert lib.softmax_debug_set(0, 0) == 0
    assert lib.softmax_sync(s) == 0                       # reported once
    assert lib.softmax_debug_set(7, 0) == 1               # unknown flags
    Y = run(lib, Xs, cols, DT_F32)
    assert lib.softmax_sync(s) == 0
    check(orc, Xs, cols, DT_F32, DT_F32, Y, canary=False)

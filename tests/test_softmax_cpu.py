"""Host logic of the row softmax, no GPU: argument checks and the work split
(include/softmax_sm103.h)."""
import pytest

import mixed_precision_dense_sm_gb300 as lib
from workloads import DT_BF16, DT_F16, DT_F32

OK, INVALID = 0, 1


def plan(rows, cols, x=256, ldx=None, xdt=DT_F32, y=1 << 44, ldy=None, ydt=DT_F32, sms=152,
         per_sm=0):
    ldx = ldx or max(cols, 1)
    ldy = ldy or max(cols, 1)
    return lib.softmax_plan_query(rows, cols, x, ldx, xdt, y, ldy, ydt, sms, per_sm)


def test_exports():
    for name in ("softmax_rows", "softmax_plan_query", "softmax_sync", "softmax_debug_set"):
        assert name in lib.declared_symbols()
        assert hasattr(lib.lib, name)


def test_argument_checks():
    assert plan(10, 10)[0] == OK
    bad = [dict(rows=-1), dict(cols=-1), dict(cols=(1 << 30) + 1), dict(ldx=9), dict(ldy=9),
           dict(xdt=5), dict(ydt=-1), dict(x=0), dict(y=0), dict(x=258), dict(y=2, ydt=DT_F32),
           dict(x=257, xdt=DT_BF16)]
    for b in bad:
        kw = dict(rows=10, cols=10)
        kw.update(b)
        assert plan(**kw)[0] == INVALID, b
    # empty problems need no pointers
    assert plan(0, 10, x=0, y=0)[0] == OK and plan(0, 10, x=0, y=0)[1]["mode_name"] == "noop"
    assert plan(10, 0, x=0, y=0)[1]["mode_name"] == "noop"
    # the raw entry point rejects the same arguments before touching a GPU
    assert lib.softmax_rows(10, 10, 0, 10, DT_F32, 256, 10, DT_F32, 0) == INVALID
    assert lib.softmax_rows(0, 10, 0, 10, DT_F32, 0, 10, DT_F32, 0) == OK


def test_overlap_rules():
    # in place: same pointer, same ld, same type
    assert plan(100, 64, x=4096, y=4096)[0] == OK
    # same pointer but another type or pitch, or a partial overlap: rejected
    assert plan(100, 64, x=4096, y=4096, ydt=DT_F16)[0] == INVALID
    assert plan(100, 64, x=4096, y=4096, ldy=72)[0] == INVALID
    assert plan(100, 64, x=4096, y=4096 + 256)[0] == INVALID
    # adjacent, not overlapping
    assert plan(100, 64, x=4096, y=4096 + 100 * 64 * 4)[0] == OK
    assert plan(100, 64, x=4096 + 100 * 64 * 4, y=4096)[0] == OK


@pytest.mark.parametrize("cols,mode,threads,cluster", [
    (1, "warp", 256, 1), (1024, "warp", 256, 1), (1025, "cta", 256, 1), (8192, "cta", 256, 1),
    (8193, "cta", 512, 1), (16384, "cta", 512, 1), (16385, "stream", 512, 1),
    (32768, "stream", 512, 1), (32769, "stream", 512, 1), (131072, "stream", 512, 2),
    (131073, "stream", 512, 2), (1 << 20, "stream", 512, 8)])
def test_work_split(cols, mode, threads, cluster):
    """Rows not 16-byte aligned (base 4 bytes off): held in registers up to
    16384 elements; longer rows in two passes by one CTA, or by a cluster
    when the slices of 152 resident CTAs would exceed 64 MB (half the L2)."""
    st, p = plan(64, cols, x=260)
    assert st == OK
    assert (p["mode_name"], p["threads"], p["cluster"]) == (mode, threads, cluster)
    assert p["slice"] % 8 == 0 and p["slice"] * p["cluster"] >= cols
    assert (p["slice"] - 8) * p["cluster"] < cols          # no CTA of the cluster is idle
    if mode != "warp":
        assert p["slice"] <= p["threads"] * 32 or mode == "stream"
        assert p["grid"] % p["cluster"] == 0
    reads = 2 if mode == "stream" else 1
    assert p["hbm_bytes"] == 64 * cols * (4 * reads + 4)
    assert p["depth"] == 0 and p["vec"] == 0


@pytest.mark.parametrize("cols,dt,ld,cl,gw,unit,depth,kv", [
    (64, DT_F32, 64, 1, 8, 32, 8, 1), (1024, DT_F32, 1024, 1, 8, 8, 3, 8),
    (1000, DT_F32, 1004, 1, 8, 8, 3, 8), (128, DT_BF16, 128, 1, 8, 32, 8, 1),
    (1024, DT_BF16, 1024, 1, 8, 8, 6, 4), (2048, DT_F32, 2048, 1, 4, 1, 6, 4),
    (4096, DT_BF16, 4096, 1, 4, 1, 6, 4), (2052, DT_F32, 2052, 1, 4, 1, 6, 8),
    (4096, DT_F32, 4096, 1, 8, 1, 6, 4), (8192, DT_F32, 8192, 1, 16, 1, 6, 4),
    (16384, DT_F32, 16384, 1, 16, 1, 3, 8), (16384, DT_BF16, 16384, 1, 16, 1, 6, 4),
    (3000, DT_F16, 3000, 1, 4, 1, 8, 4), (8192, DT_BF16, 8192, 1, 8, 1, 6, 4),
    (2048, DT_BF16, 2048, 1, 8, 8, 3, 8), (1536, DT_F16, 1536, 1, 8, 8, 4, 8),
    (32768, DT_F16, 32768, 1, 16, 1, 3, 8), (20000, DT_BF16, 20000, 1, 16, 1, 5, 8),
    # too long to stage whole: streamed twice in 32 KB chunks (6 slots, the
    # CTA's 16 warps on one row, 4 vectors per thread per chunk), the row
    # split over a cluster of 2-8 CTAs when the slices of 152 SMs would
    # exceed 64 MB of L2
    (16388, DT_F32, 16388, 1, 16, 1, 6, 4), (32776, DT_F16, 32776, 1, 16, 1, 6, 4),
    (65536, DT_F32, 65536, 1, 16, 1, 6, 4), (110376, DT_F32, 110376, 1, 16, 1, 6, 4),
    (131072, DT_F32, 131072, 2, 16, 1, 6, 4), (110384, DT_F32, 110384, 2, 16, 1, 6, 4),
    (131080, DT_F32, 131080, 2, 16, 1, 6, 4), (1 << 20, DT_F32, 1 << 20, 8, 16, 1, 6, 4),
    (300001 + 7, DT_BF16, 300008, 2, 16, 1, 6, 4),
    # not staged: too short, or rows not 16-byte aligned
    (60, DT_F32, 60, 1, 0, 0, 0, 0), (120, DT_BF16, 120, 1, 0, 0, 0, 0),
    (16385, DT_F32, 16385, 1, 0, 0, 0, 0)])
def test_staged_split(cols, dt, ld, cl, gw, unit, depth, kv):
    """16-byte-aligned rows of 256 B to 64 KB and at most 16 x 32 x 8
    16-byte vectors (16384 FP32 or 32768 16-bit elements) are staged in
    shared memory by bulk copies: one CTA of 16 compute warps and a producer
    warp per SM.  Rows a warp can hold (<= 8 vectors per thread: 256 FP32 or
    2048 16-bit elements) go to groups of 8 warps whose slots carry several
    rows (~16 KB, one copy when the rows are adjacent), a warp per row;
    longer rows are shared by the smallest group that holds them in
    registers, doubled while a group would get fewer than six slots.  Each group is a
    pipeline with as many slots as 200 KB allow (at most 8).  Other rows keep
    the register kernels (depth 0)."""
    st, p = plan(100000, cols, ldx=ld, ldy=ld, xdt=dt, ydt=dt)
    assert st == OK
    got = (p["cluster"], p["group_warps"], p["unit_rows"], p["depth"], p["kv"])
    assert got == (cl, gw, unit, depth, kv), p
    es = 4 if dt == DT_F32 else 2
    kvmax = 8                               # 16-byte vectors per thread
    if depth and p["mode_name"] == "stream":
        # long rows: a 32 KB chunk per slot, X read twice (the second time
        # from L2); a cluster's CTAs take equal slices, multiples of 8
        assert p["vec"] == 1 and p["threads"] == 544 and p["grid"] == cl * (152 // cl)
        assert cols * es > 64 * 1024
        sl = p["slice"]
        assert sl % 8 == 0 and sl * cl >= cols and (sl - 8) * cl < cols
        assert 152 * sl * es <= 64 << 20 or cl == 8
        assert cl == 1 or 152 * -(-cols // (cl // 2)) * es > 64 << 20
        assert p["hbm_bytes"] == 100000 * cols * 3 * es
        assert plan(5, cols, ldx=ld, ldy=ld, xdt=dt, ydt=dt)[1]["grid"] == 5 * cl
        return
    if depth:
        assert p["vec"] == 1 and p["threads"] == 544          # 16 compute warps + the producer
        assert p["grid"] == (152 if cl == 1 else cl * (152 // cl))
        assert p["mode_name"] == ("warp" if unit > 1 else "cta")
        groups = 16 // gw
        slice_ = p["slice"] if cl > 1 else cols
        assert slice_ % 8 == 0 or cl == 1
        assert cl == 1 or ((cols + cl - 1) // cl <= slice_ < (cols + cl - 1) // cl + 8)
        stride = ld * es if unit > 1 else slice_ * es
        slot = -(-unit * stride // 128) * 128
        assert groups * depth * slot <= 200 * 1024 and depth >= 3
        nvec = slice_ * es // 16
        if unit == 1:
            assert gw * 32 * kvmax >= nvec
            # the fewest warps that hold the row, unless half as many would
            # leave a group fewer than six slots
            assert cl > 1 or gw == 1 or (gw // 2) * 32 * kvmax < nvec or \
                (16 // (gw // 2)) * 6 * slot > 200 * 1024
            assert kv * gw * 32 >= nvec and (kv == 1 or (kv // 2) * gw * 32 < nvec)
        else:
            assert nvec <= 32 * kvmax and unit % gw == 0
            assert kv * 32 >= nvec and (kv == 1 or (kv // 2) * 32 < nvec)
        assert p["hbm_bytes"] == 100000 * cols * 2 * es
        if cl == 1:
            rows = 5 * unit
            assert plan(rows, cols, ldx=ld, ldy=ld, xdt=dt, ydt=dt)[1]["grid"] == -(-5 // groups)
        else:
            assert plan(3, cols, ldx=ld, ldy=ld, xdt=dt, ydt=dt)[1]["grid"] == 3 * cl
    few = plan(3, cols, xdt=dt, ydt=dt)[1]
    assert few["grid"] <= 3 * few["cluster"]


def test_vector_rule_and_grid():
    assert plan(8, 4096)[1]["vec"] == 1
    assert plan(8, 4096, ldx=4097)[1]["vec"] == 0               # FP32 rows 4 B apart
    assert plan(8, 4096, xdt=DT_BF16, ldx=4100)[1]["vec"] == 0  # 16-bit rows need ld % 8
    assert plan(8, 4096, xdt=DT_BF16, ldx=4104)[1]["vec"] == 1
    assert plan(8, 4096, x=260)[1]["vec"] == 0                  # base not 16-byte aligned
    # persistent grids: never more groups than rows, nor than resident groups
    assert plan(3, 100, x=260)[1]["grid"] == 1                    # 8 rows per CTA
    assert plan(100000, 100, x=260, per_sm=2)[1]["grid"] == 2 * 152
    assert plan(5, 4096, x=260, per_sm=2)[1]["grid"] == 5
    assert plan(100000, 4096, x=260, per_sm=2)[1]["grid"] == 304
    assert plan(100000, 100)[1]["grid"] == 152                    # staged: one CTA per SM
    assert plan(100000, 65536, per_sm=10)[1]["grid"] == 152       # long rows: one CTA per SM
    assert plan(100, 65536)[1]["grid"] == 100
    assert plan(100000, 65536, x=260, per_sm=10)[1]["grid"] == 10 * 152  # two passes, a CTA per row
    assert plan(100000, 1 << 20, per_sm=10)[1]["grid"] == 8 * 10  # 10 clusters of 8


def test_plan_invariants_on_random_rows():
    """Seeded random shapes, types and alignments: each plan's kind follows
    from the row (staged when 16-byte aligned, 256 B to 64 KB and at most
    16 x 32 x 8 vectors; long rows streamed twice when aligned and longer,
    on clusters that keep 152 slices within 64 MB of L2; register kernels
    otherwise), its threads hold the whole row, its slots fit the 200 KB
    budget, and its HBM bytes count X twice exactly when it reads X twice."""
    import random
    rng = random.Random(7919)
    kinds = {"staged": 0, "long": 0, "register": 0}
    for _ in range(600):
        xdt, ydt = rng.choice([DT_F32, DT_F16, DT_BF16]), rng.choice([DT_F32, DT_F16, DT_BF16])
        ex, ey = (4 if xdt == DT_F32 else 2), (4 if ydt == DT_F32 else 2)
        cols = rng.choice([rng.randint(1, 4096), rng.randint(4096, 40000), rng.randint(40000, 400000)])
        rows = rng.randint(1, 3000)
        aligned = rng.random() < 0.7
        ldx = cols + (-cols) % 8 if aligned else cols + rng.randint(0, 3)
        ldy = cols + (-cols) % 8 if aligned else cols
        x = 256 if aligned else 256 + rng.choice([0, ex])
        st, p = plan(rows, cols, x=x, ldx=ldx, xdt=xdt, ldy=ldy, ydt=ydt)
        assert st == OK
        vec = (x % 16 == 0) and (ldx * ex) % 16 == 0 and (ldy * ey) % 16 == 0
        assert p["vec"] == (1 if vec else 0)
        b = cols * ex
        staged = vec and 256 <= b <= 64 * 1024 and b // 16 <= 16 * 32 * 8
        if staged:
            kinds["staged"] += 1
            assert p["depth"] > 0 and p["mode_name"] in ("warp", "cta") and p["threads"] == 544
            gw, unit, kv = p["group_warps"], p["unit_rows"], p["kv"]
            assert gw in (1, 2, 4, 8, 16) and kv in (1, 2, 4, 8)
            nvec = b // 16
            holders = 32 if unit > 1 else 32 * gw
            assert kv * holders >= nvec and (kv == 1 or (kv // 2) * holders < nvec)
            assert p["hbm_bytes"] == rows * cols * (ex + ey)
        elif vec and cols > 16384 and p["cluster"] <= 8 and p["depth"] > 0:
            kinds["long"] += 1
            cl, sl = p["cluster"], p["slice"]
            assert p["mode_name"] == "stream" and p["depth"] == 6 and p["kv"] == 4
            assert sl % 8 == 0 and sl * cl >= cols and (sl - 8) * cl < cols
            assert cl == 1 or 152 * -(-cols // (cl // 2)) * ex > 64 << 20
            assert p["hbm_bytes"] == rows * cols * (2 * ex + ey)
        else:
            kinds["register"] += 1
            assert p["depth"] == 0
            assert not vec or cols <= 16384 or b < 256, (rows, cols, xdt, ydt, p)
            reads = 2 if p["mode_name"] == "stream" else 1
            assert p["hbm_bytes"] == rows * cols * (reads * ex + ey)
    assert min(kinds.values()) > 30, kinds

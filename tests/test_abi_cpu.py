"""The C ABI library on the CPU: it loads, exports every symbol the header
declares, validates arguments and plans paths (host logic only, no GPU)."""
import ctypes
import math
import itertools
import subprocess

import pytest
import torch

import mixed_precision_dense_sm_gb300 as lib
import workloads
from workloads import DT_BF16, DT_F16, DT_F32

F16F32 = (DT_F16, DT_F16, DT_F32)
TF32 = (DT_F32, DT_F32, DT_F32)


def test_exports_every_declared_symbol():
    declared = lib.declared_symbols()
    assert declared == sorted(["gemm_check_args", "gemm_create", "gemm_destroy",
                               "gemm_plan_query", "gemm_run", "gemm_status_string",
                               "gemm_sync"]) or set(declared) >= {"gemm_create", "gemm_run"}
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for name in declared:
        assert name in exported, name
        assert hasattr(lib.lib, name)


def test_debug_hook_validates_arguments():
    assert lib.gemm_debug_set(None, 0, 0) == 1
    assert lib.GEMM_DEBUG_SKIP_FIRST_LOAD == 1
    assert "gemm_debug_set" in lib.declared_symbols()


def test_status_strings():
    for code, name in lib.STATUS.items():
        assert lib.gemm_status_string(code) == name
    assert lib.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


def test_check_args():
    ok = dict(ta="N", tb="N", M=8, N=8, K=8, alpha=1.0, A=16, lda=8, B=16, ldb=8, beta=0.0,
              C=16, ldc=8, dt=F16F32)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.gemm_check_args(a["ta"], a["tb"], a["M"], a["N"], a["K"], a["alpha"], a["A"],
                                   a["lda"], a["B"], a["ldb"], a["beta"], a["C"], a["ldc"],
                                   a["dt"])

    assert call() == 0
    assert call(ta="t", tb="n") == 0
    for bad in [dict(ta="X"), dict(tb="?"), dict(M=-1), dict(N=-2), dict(K=-3),
                dict(lda=7), dict(ldb=7), dict(ldc=7), dict(ta="T", lda=7, M=8),
                dict(tb="T", ldb=7), dict(dt=(DT_F16, DT_BF16, DT_F32)),
                dict(dt=(DT_F32, DT_F16, DT_F32)), dict(dt=(DT_BF16, DT_F32, DT_F32)),
                dict(dt=(DT_F16, DT_F16, 5)), dict(dt=(3, 3, DT_F32)),
                dict(A=0), dict(B=0), dict(C=0), dict(M=2 ** 31),
                # each pointer aligned to its own element size
                dict(A=17), dict(B=19), dict(C=18), dict(C=17, dt=(DT_F16, DT_F16, DT_F16)),
                dict(A=18, dt=TF32), dict(B=22, dt=TF32)]:
        assert call(**bad) == 1, bad
    # FP32 inputs are computed as TF32
    assert call(dt=TF32) == 0
    assert call(dt=(DT_F32, DT_F32, DT_BF16), C=18) == 0
    assert call(A=18, B=30) == 0                     # 2-byte aligned FP16 operands
    # quick-return forms
    assert call(M=0, C=0, A=0, B=0) == 0
    assert call(K=0, A=0, B=0) == 0
    assert call(alpha=0.0, A=0, B=0) == 0
    assert call(alpha=0.0, A=17, B=17) == 0          # A and B are not read
    assert call(K=0, lda=1) == 0


def plan(w: workloads.Workload, ptr=256, **kw):
    lda, ldb, ldc = w.lds()
    st, p = lib.gemm_plan_query(w.transA, w.transB, w.M, w.N, w.K, w.alpha, ptr, lda, ptr, ldb,
                                w.beta, ptr, ldc, (w.ab_dtype, w.ab_dtype, w.c_dtype), **kw)
    assert st == 0
    return p


def test_plans_of_named_workloads():
    P = {n: plan(w) for n, w in workloads.WORKLOADS.items()}
    big = P["linear_8192x4096x4096_bf16"]
    assert big["path_name"] == "tiled_2sm" and big["block_n"] == 256 and big["sk_len"] == 0
    assert big["block_m"] == 256 and big["grid"] == 152 and big["num_tiles"] == 32 * 16
    for n in ("linear_8192x14336x4096_bf16", "linear_8192x4096x14336_bf16"):
        assert P[n]["path_name"] == "tiled_2sm" and P[n]["grid"] % 2 == 0
    sk = P["skinny_64x16384x8192_f16"]
    assert sk["path_name"] == "skinny" and sk["swap_ab"] == 1 and sk["block_n"] == 64
    rag = P["ragged1000x1023x777_bf16_beta1"]
    assert rag["pack_a"] == 1 and rag["pack_b"] == 1 and rag["c_vector"] == 0
    assert rag["b_mn_major"] == 1 and rag["a_mn_major"] == 0
    sq = P["square1024_f16_nt_f16out"]
    assert sq["pack_a"] == 0 and sq["pack_b"] == 0 and sq["b_mn_major"] == 0
    for n, p in P.items():
        assert 2 <= p["stages"] <= 8
        cg = p["block_m"] // 128
        esize = 4 if workloads.WORKLOADS[n].ab_dtype == DT_F32 else 2
        # one or two 128-byte swizzle rows (chunks) of K per stage
        kc = p["block_k"] * esize // 128
        assert p["block_k"] * esize in (128, 256)
        assert p["k_blocks"] == -(-workloads.WORKLOADS[n].K // p["block_k"])
        stage = kc * (128 * 128 + (p["block_n"] // cg) * 128)
        assert p["stages"] * stage + 1024 + 256 <= 232448
        if kc == 2:
            assert p["stages"] >= 3


def test_two_k_chunks_per_stage():
    """Two 128-byte rows of K per stage (half the TMA boxes per MMA) whenever
    a K-major operand's K is a whole number of chunks and 3 stages fit;
    otherwise one (a 3-D view would read past the row's end)."""
    def p(ta, tb, M, N, K, dt=(DT_BF16, DT_BF16, DT_BF16)):
        lda = K if ta == "N" else M
        ldb = K if tb == "T" else N
        st, q = lib.gemm_plan_query(ta, tb, M, N, K, 1.0, 256, lda, 256, ldb, 0.0, 256, N, dt)
        assert st == 0
        return q
    assert p("N", "T", 8192, 4096, 4096)["block_k"] == 128           # CTA pairs: 3 x 64 KB
    assert p("N", "T", 1024, 1024, 1024)["block_k"] == 128
    assert p("N", "T", 1024, 1024, 1000)["block_k"] == 64            # K not a whole chunk
    assert p("T", "N", 1024, 1024, 1000)["block_k"] == 128           # both MN-major: zero fill
    assert p("N", "N", 1024, 1024, 1000)["block_k"] == 64            # A K-major
    q = p("N", "T", 200, 3072, 4096)                                 # 1-SM 256 wide: 2 x 96 KB
    assert (q["path_name"], q["block_n"], q["block_k"]) == ("tiled_1sm", 256, 64), q
    q = p("N", "T", 512, 3072, 4096)                                 # CTA pairs, stream-K
    assert (q["path_name"], q["block_n"], q["block_k"]) == ("tiled_2sm", 256, 128), q
    assert p("N", "T", 100, 100, 128, (DT_F32, DT_F32, DT_F32))["block_k"] == 64   # TF32: 2 x 32
    # strided convolutions (im2col tiles): two chunks (two im2col boxes, one
    # filter box) when C is a whole number of 64-channel blocks; 9 taps x 1
    # block = 9 chunks, 5 stages
    st, c = lib.conv2d_plan_query(32, 112, 112, 64, 64, 3, 3, (1, 1), (2, 2), (1, 1), 1.0, 256, 256,
                                  0.0, 256, (DT_BF16, DT_BF16, DT_BF16))
    assert st == 0 and c["block_k"] == 128 and c["k_blocks"] == 5, c
    st, c = lib.conv2d_plan_query(8, 40, 40, 96, 64, 3, 3, (1, 1), (2, 2), (1, 1), 1.0, 256, 256,
                                  0.0, 256, (DT_BF16, DT_BF16, DT_BF16))
    assert st == 0 and c["block_k"] == 64 and c["k_blocks"] == 18, c
    # a convolution on single-CTA 256-wide tiles keeps two chunks in two
    # stages (operands re-read from L2); a GEMM of that tile keeps one chunk
    st, c = lib.conv2d_plan_query(1, 14, 14, 64, 19456, 3, 3, (1, 1), (1, 1), (1, 1), 1.0, 256, 256,
                                  0.0, 256, (DT_BF16, DT_BF16, DT_BF16))
    assert st == 0 and (c["path_name"], c["block_n"], c["block_k"], c["stages"]) == \
        ("tiled_1sm", 256, 128, 2), c
    # the 14 x 14 layer, C = K = 512: too few pair tiles, long K -> stream-K on CTA pairs
    st, c = lib.conv2d_plan_query(32, 14, 14, 512, 512, 3, 3, (1, 1), (1, 1), (1, 1), 1.0, 256, 256,
                                  0.0, 256, (DT_BF16, DT_BF16, DT_BF16))
    assert st == 0 and (c["path_name"], c["block_n"], c["block_k"], c["stages"]) == \
        ("tiled_2sm", 256, 128, 3) and c["sk_len"] > 0, c


def test_quick_paths_and_swap_rule():
    w = workloads.Workload("q", 0, 5, 5, "N", "N", DT_F16, DT_F32, 1.0, 0.0, "U", "U")
    assert plan(w)["path_name"] == "noop"
    w = workloads.Workload("q", 5, 5, 0, "N", "N", DT_F16, DT_F32, 1.0, 1.0, "U", "U", "U")
    assert plan(w)["path_name"] == "scale"
    w = workloads.Workload("q", 5, 5, 5, "N", "N", DT_F16, DT_F32, 0.0, 1.0, "U", "U", "U")
    assert plan(w)["path_name"] == "scale"
    w = workloads.Workload("q", 64, 128, 64, "N", "N", DT_F16, DT_F32, 1.0, 0.0, "U", "U")
    assert plan(w)["swap_ab"] == 1
    w = workloads.Workload("q", 65, 128, 64, "N", "N", DT_F16, DT_F32, 1.0, 0.0, "U", "U")
    assert plan(w)["swap_ab"] == 0


@pytest.mark.parametrize("N,K,swapped", [(16384, 8192, False), (4096, 4096, False),
                                         (14336, 4096, True), (14336, 1024, False),
                                         (8192, 8192, False)])
def test_decode_batches_up_to_128_rows(N, K, swapped):
    """64 < M <= 128 (one tile row): swapped only when the unswapped plan's
    single wave of 128-wide tiles would be under 80 % full and long in K
    (then balanced by stream-K over 256-wide tiles, which the swapped stream-K
    beats); M <= 64 always swaps, M > 128 never."""
    for M in (80, 96, 112, 128):
        w = workloads.Workload("d", M, N, K, "N", "T", DT_F16, DT_F16, 1.0, 0.0, "N1", "N002")
        p = plan(w)
        assert p["swap_ab"] == (1 if swapped else 0), (M, p)
        assert p["path_name"] == ("skinny" if swapped else "tiled_1sm")
    for M, want in ((64, 1), (129, 0)):
        w = workloads.Workload("d", M, N, K, "N", "T", DT_F16, DT_F16, 1.0, 0.0, "N1", "N002")
        assert plan(w)["swap_ab"] == want


def test_pair_tiles_only_when_they_fill_the_gpu():
    def path(M, N, K, sms=152):
        w = workloads.Workload("p", M, N, K, "N", "T", DT_BF16, DT_BF16, 1.0, 0.0, "U", "U")
        return plan(w, num_sms=sms)
    assert path(4096, 4096, 4096)["path_name"] == "tiled_2sm"     # 256 pair tiles
    assert path(2048, 2048, 4096)["path_name"] == "tiled_1sm"     # 64 pair tiles < 76 pairs
    p = path(2048, 4864, 1024)                                    # 8 x 19 = 152 >= 76
    assert p["path_name"] == "tiled_2sm" and p["grid"] == 152
    p = path(300, 100000, 64, sms=8)
    assert p["path_name"] == "tiled_2sm" and p["grid"] == 8


def test_pack_rule_follows_16_byte_alignment():
    w = workloads.Workload("p", 100, 100, 100, "N", "N", DT_F16, DT_F32, 1.0, 0.0, "U", "U",
                           lda=104, ldb=100 + 3)
    p = plan(w)
    assert p["pack_a"] == 0 and p["pack_b"] == 1
    p = plan(w, ptr=260)          # misaligned base: everything packs, C scalar path
    assert p["pack_a"] == 1 and p["pack_b"] == 1 and p["c_vector"] == 0


def test_tf32_plans():
    """FP32 inputs (TF32): chunks of 32 elements of K (two per stage when K
    is a whole number of chunks), the same tile shapes and rules as 16-bit
    inputs, packing when rows are not 16-byte aligned (a pitch that is not a
    multiple of 4 elements)."""
    w = workloads.WORKLOADS["tf32_linear_8192x4096x4096_f32out"]
    p = plan(w)
    assert p["path_name"] == "tiled_2sm" and p["block_k"] == 64 and p["k_blocks"] == 64
    assert p["pack_a"] == 0 and p["pack_b"] == 0
    w = workloads.Workload("t", 100, 100, 100, "N", "N", DT_F32, DT_F32, 1.0, 0.0, "U", "U",
                           lda=104, ldb=102)
    p = plan(w)
    assert p["pack_a"] == 0 and p["pack_b"] == 1 and p["k_blocks"] == 4
    p = plan(w, ptr=260)          # 4-byte but not 16-byte aligned base: everything packs
    assert p["pack_a"] == 1 and p["pack_b"] == 1 and p["c_vector"] == 0
    w = workloads.Workload("t", 64, 16384, 8192, "N", "T", DT_F32, DT_F32, 1.0, 0.0, "U", "U")
    p = plan(w)
    assert p["path_name"] == "skinny" and p["sk_len"] > 0 and p["k_blocks"] == 128
    # the same rules as the 16-bit path, for every tile width
    for M, N, K in [(1000, 1023, 777), (4096, 4096, 4096), (257, 129, 4096), (64, 1000, 513)]:
        a = plan(workloads.Workload("t", M, N, K, "N", "N", DT_F32, DT_F32, 1.0, 0.0, "U", "U",
                                    lda=K + 4, ldb=N + 4))
        b = plan(workloads.Workload("h", M, N, K, "N", "N", DT_F16, DT_F32, 1.0, 0.0, "U", "U",
                                    lda=K + 8, ldb=N + 8))
        for key in ("path_name", "block_m", "block_n", "swap_ab", "tiles_m", "tiles_n"):
            assert a[key] == b[key], (M, N, K, key)
        assert a["k_blocks"] == -(-K // a["block_k"]) and a["block_k"] in (32, 64)


def test_tf32_operands_stored_mn_major_are_transposed_first():
    """kind::tf32 reads K-major operands only: an FP32 operand stored with
    M or N contiguous (A with 'T', B with 'N') is rewritten K-contiguous by a
    pre-pass into the workspace; 16-bit operands never are."""
    M, N, K = 300, 400, 500
    for ta, tb, want in [("N", "T", 0), ("N", "N", 2), ("T", "T", 1), ("T", "N", 3)]:
        p = plan(workloads.Workload("t", M, N, K, ta, tb, DT_F32, DT_F32, 1.0, 0.0, "U", "U"))
        assert p["transpose_ab"] == want, (ta, tb, p)
        assert p["a_mn_major"] == 0 and p["b_mn_major"] == 0
        assert p["pack_a"] == (want & 1) and p["pack_b"] == (want >> 1)
        need = (M * 500 if want & 1 else 0) * 4 + (N * 500 if want & 2 else 0) * 4
        assert p["workspace_bytes"] >= need
        h = plan(workloads.Workload("h", M, N, K, ta, tb, DT_BF16, DT_F32, 1.0, 0.0, "U", "U"))
        assert h["transpose_ab"] == 0
        assert h["a_mn_major"] == (ta == "T") and h["b_mn_major"] == (tb == "N")
    # the swapped skinny path reports the user's operands
    p = plan(workloads.Workload("s", 32, 4096, 512, "N", "N", DT_F32, DT_F32, 1.0, 0.0, "U", "U"))
    assert p["swap_ab"] == 1 and p["transpose_ab"] == 2 and p["pack_b"] == 1 and p["pack_a"] == 0
    p = plan(workloads.Workload("s", 32, 4096, 512, "T", "T", DT_F32, DT_F32, 1.0, 0.0, "U", "U"))
    assert p["swap_ab"] == 1 and p["transpose_ab"] == 1 and p["pack_a"] == 1 and p["pack_b"] == 0


def simulate_stream_k(p):
    """Replays the device-side segment iteration for every CTA and checks the
    schedule: each (tile, k-block) is covered exactly once, partial slots are
    unique and in range, the finisher's slot lookup finds the same slots, and
    the finisher of every split tile (the CTA holding its first k-blocks) meets
    it in the last segment of its range -- so its other TMEM buffer is free
    for the pre-summed partials and it is the contributor that ends last."""
    cg = 2 if p["path_name"] == "tiled_2sm" else 1          # CTAs per unit (a pair shares a range)
    assert p["grid"] % cg == 0
    T, KB, L, G, S = p["num_tiles"], p["k_blocks"], p["sk_len"], p["grid"] // cg, p["sk_max_seg"]
    total = T * KB
    covered = [0] * total
    slots = {}
    last_tile = {}
    for g in range(G):
        pos, end = min(g * L, total), min(g * L + L, total)
        assert pos < end, "a CTA without work"
        while pos < end:
            tile = pos // KB
            last_tile[g] = tile
            kb0 = pos - tile * KB
            take = min(KB - kb0, end - pos)
            for k in range(kb0, kb0 + take):
                covered[tile * KB + k] += 1
            pos += take
            if not (kb0 == 0 and take == KB):
                first_tile = (g * L) // KB
                slot = g * S + (tile - first_tile)
                assert 0 <= tile - first_tile < S
                assert slot not in slots
                slots[slot] = (tile, g)
    assert all(c == 1 for c in covered)
    for tile in range(T):
        g_first, g_last = (tile * KB) // L, ((tile + 1) * KB - 1) // L
        if g_first == g_last:
            continue
        for g in range(g_first, g_last + 1):
            slot = g * S + tile - (g * L) // KB
            assert slots.get(slot) == (tile, g)
        assert last_tile[g_first] == tile
    assert T * cg <= 1024             # one int32 counter per tile and CTA in the 4 KB header
    assert len(slots) * p["block_m"] * p["block_n"] * 4 <= p["workspace_bytes"]


@pytest.mark.parametrize("shape", [(256, 256, 256), (1024, 1024, 1024), (1000, 1023, 777),
                                   (64, 16384, 8192), (5, 300, 700), (129, 300, 777),
                                   (257, 129, 4096), (33, 128, 2048), (1, 1, 100000),
                                   (6272, 512, 4608), (25088, 256, 4096), (9000, 700, 3000)])
@pytest.mark.parametrize("sms", [148, 152, 7])
def test_stream_k_schedule_covers_every_block_once(shape, sms):
    M, N, K = shape
    w = workloads.Workload("s", M, N, K, "N", "T", DT_BF16, DT_BF16, 1.0, 0.0, "U", "U")
    p = plan(w, num_sms=sms)
    if p["sk_len"] == 0:
        return                      # data-parallel plan: nothing to replay
    assert p["grid"] <= sms
    simulate_stream_k(p)


def test_stream_k_only_for_skinny_tile_starved_or_badly_filled_long_k():
    def P(M, N, K, sms=152):
        w = workloads.Workload("s", M, N, K, "N", "T", DT_BF16, DT_BF16, 1.0, 0.0, "U", "U")
        return plan(w, num_sms=sms)
    assert P(64, 16384, 8192)["sk_len"] > 0          # swapped weight-streaming GEMM
    assert P(257, 129, 4096)["sk_len"] > 0           # 6 tiles, 64 k-blocks each
    assert P(1, 1, 100000)["sk_len"] > 0
    # data-parallel waves filled below 80 % with 32+ k-blocks per tile: stream-K
    # over the widest single-CTA tiles, possibly more tiles than SMs
    # over the widest tiles, on CTA pairs when M has 256 rows
    p = P(6272, 512, 4608)                           # 196 tiles of 128 x 128: 1.29 waves
    assert p["sk_len"] > 0 and p["block_n"] == 256 and p["path_name"] == "tiled_2sm"
    p = P(25088, 256, 4096)                          # 98 CTA-pair tiles on 76 pairs
    assert p["sk_len"] > 0 and p["num_tiles"] == 98 and p["grid"] <= 152
    assert p["path_name"] == "tiled_2sm"
    p = P(200, 3072, 4096)                           # 24 tiles, fewer than 256 rows: single CTAs
    assert p["sk_len"] > 0 and p["block_n"] == 256 and p["path_name"] == "tiled_1sm"
    assert P(25088, 128, 1152)["sk_len"] == 0        # same fill, 18 k-blocks: not worth it
    assert P(65536, 256, 2304)["path_name"] == "tiled_2sm"   # 256 pair tiles: 84 % fill
    for shape in [(1024, 1024, 1024), (1000, 1023, 777), (256, 256, 256), (300, 520, 1000)]:
        assert P(*shape)["sk_len"] == 0, shape
    assert P(1024, 1024, 1024)["block_n"] == 64      # 128 tiles of 128 x 64
    assert P(256, 256, 256)["num_tiles"] >= 4


@pytest.mark.parametrize("shape", [(256, 256, 2048), (2048, 256, 4096), (300, 2048, 4096),
                                   (512, 3072, 4096), (6272, 512, 4608), (1536, 2048, 14336),
                                   (200, 3072, 4096), (257, 129, 4096), (33, 128, 2048)])
def test_stream_k_split_is_capped(shape):
    """A tile split s ways saves (1 - 1/s) of its K loop and costs its finisher
    s - 1 partial tiles read back, each worth about 8 k-blocks of 256-byte rows:
    ranges are at least k_blocks / floor(sqrt(k_blocks / 8)) long (the skinny
    weight-streaming path excepted), so no tile has more contributors than
    that bound plus one."""
    M, N, K = shape
    w = workloads.Workload("s", M, N, K, "N", "T", DT_BF16, DT_BF16, 1.0, 0.0, "U", "U")
    p = plan(w)
    KB, L = p["k_blocks"], p["sk_len"]
    fixup = 8.0 * 256 / (p["block_k"] * 2)
    s_max = max(1, int(math.floor(math.sqrt(KB / fixup))))
    if L and p["path_name"] != "skinny":
        assert L >= -(-KB // s_max), p
        for tile in range(p["num_tiles"]):
            assert ((tile + 1) * KB - 1) // L - (tile * KB) // L + 1 <= s_max + 1
    if shape == (256, 256, 2048):                    # 16 k-blocks: never split
        assert L in (0, KB), p


def test_tma_store_of_c_where_it_pays():
    """C goes through shared memory and TMA stores when its rows are 16-byte
    aligned, beta == 0 and either C is FP32 with K >= 2048 or each CTA (pair)
    gets two or more data-parallel tiles; never for the swapped skinny path or
    LayerNorm, and the staging never costs a pipeline stage."""
    def q(M, N, K, c=DT_BF16, beta=0.0, ldc=None, ab=DT_BF16):
        st, p = lib.gemm_plan_query("N", "T", M, N, K, 1.0, 256, K, 256, K, beta, 256,
                                    ldc or N, (ab, ab, c), num_sms=152)
        assert st == 0
        return p
    assert q(8192, 4096, 4096)["c_tma"] == 1                  # 512 pair tiles on 76 pairs
    assert q(8192, 4096, 4096)["stages"] == 3
    assert q(8192, 4096, 4096, beta=1.0)["c_tma"] == 0        # residual: row stores
    assert q(8192, 4096, 4096, c=DT_F32)["c_tma"] == 1
    assert q(1024, 1024, 1024, c=DT_F16)["c_tma"] == 0        # 128 tiles: one wave
    assert q(1024, 1024, 1024, c=DT_F32)["c_tma"] == 0        # FP32, short K
    assert q(1024, 1024, 2048, c=DT_F32)["c_tma"] == 1        # FP32, K >= 2048
    assert q(6272, 512, 4608)["c_tma"] == 0                   # stream-K, 16-bit C
    assert q(512, 3072, 4096, c=DT_F32)["c_tma"] == 1         # stream-K, FP32 C
    assert q(64, 16384, 8192, c=DT_F16, ab=DT_F16)["c_tma"] == 0   # swapped
    assert q(8192, 4096, 4096, ldc=4100)["c_tma"] == 0        # rows not 16-byte aligned
    st, p = _ln_plan(8192, 4096, 4096)
    assert st == 0 and p["c_tma"] == 0


def test_create_fails_cleanly_without_gpu():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(1234)
    st = lib.lib.gemm_create(ctypes.byref(h))
    assert st in (2, 4) and h.value is None
    assert lib.gemm_destroy(None) == 0
    assert lib.gemm_sync(None, None) == 1
    assert lib.gemm_run(None, "N", "N", 1, 1, 1, 1.0, 16, 1, 16, 1, 0.0, 16, 1, F16F32) == 1


# ------------------------------------------------ LayerNorm after the linear layer

def _ln_plan(M, N, K, dts=(DT_BF16, DT_BF16, DT_BF16), num_sms=152, **kw):
    args = dict(bias=0x100, bias_dtype=DT_BF16, gamma=0x100, shift=0x100, ln_dtype=DT_F32,
                eps=1e-5)
    args.update(kw)
    return lib.gemm_layernorm_plan_query("N", "T", M, N, K, 1.0, 0x100, K, 0x100, K, 1.0, 0x100,
                                         N, dts, num_sms=num_sms, **args)


def test_layernorm_plan_whole_rows_fused():
    """Rows of up to 256 columns are normalised inside the epilogue: one tile
    column, no stream-K, never the swapped skinny path."""
    for M, N, K, path, bn in [(300, 100, 200, "tiled_1sm", 128), (517, 256, 333, "tiled_1sm", 256),
                              (40, 200, 8192, "tiled_1sm", 256),
                              (20000, 256, 192, "tiled_2sm", 256),
                              (20000, 128, 192, "tiled_1sm", 128)]:
        st, p = _ln_plan(M, N, K)
        assert st == 0, (M, N, K)
        assert p["ln_fused"] == 1 and p["tiles_n"] == 1, p
        assert (p["path_name"], p["block_n"]) == (path, bn), (M, N, K, p)
        assert p["sk_len"] == 0 and p["swap_ab"] == 0, p


def test_layernorm_plan_row_pass():
    """Wider rows: per-tile (mean, M2) in the workspace, 8 bytes per row and
    tile column; tiles of 128 or 256 columns; no stream-K even for long K."""
    for M, N, K in [(333, 1000, 500), (40, 3000, 700), (8192, 4096, 4096), (64, 16384, 8192),
                    (8192, 1024, 320)]:
        st, p = _ln_plan(M, N, K)
        assert st == 0
        assert p["ln_fused"] == 0 and p["tiles_n"] >= 2, p
        assert p["block_n"] in (128, 256) and p["sk_len"] == 0 and p["swap_ab"] == 0, p
        assert p["workspace_bytes"] >= M * p["tiles_n"] * 8, p
        st, q = lib.gemm_plan_query("N", "T", M, N, K, 1.0, 0x100, K, 0x100, K, 1.0, 0x100, N,
                                    (DT_BF16, DT_BF16, DT_BF16))
        assert st == 0


def test_layernorm_plan_rejects():
    assert _ln_plan(64, 64, 64, eps=0.0)[0] == 1
    assert _ln_plan(64, 64, 64, eps=-1e-5)[0] == 1
    assert _ln_plan(64, 64, 64, eps=float("nan"))[0] == 1
    assert _ln_plan(64, 64, 64, eps=float("inf"))[0] == 1
    assert _ln_plan(64, 64, 64, ln_dtype=5)[0] == 1
    assert _ln_plan(64, 64, 64, bias_dtype=-1)[0] == 1
    # without gamma and shift their dtype is not read
    assert _ln_plan(64, 64, 64, gamma=0, shift=0, ln_dtype=5)[0] == 0
    assert _ln_plan(64, 64, 64, dts=TF32)[0] == 2
    plan = lib.Plan()
    assert lib.lib.gemm_layernorm_plan_query(b"N", b"T", 64, 64, 64, 1.0, 0x100, 64, 0x100, 64,
                                             0.0, 0x100, 64, lib.Dtypes(0, 0, 0), None, 152,
                                             232448, ctypes.byref(plan), None) == 1
    # the GEMM's own checks still apply
    assert _ln_plan(-1, 64, 64)[0] == 1
    st, p = _ln_plan(0, 64, 64)
    assert st == 0 and p["path_name"] == "noop"


def test_plan_invariants_on_random_problems():
    """Seeded random GEMMs (shape, transposes, types, pointer and pitch
    alignment, beta, SM count): every plan's tiles cover the (possibly
    swapped) output once, the grid fits the SMs, the K loop is whole, operands
    whose rows TMA cannot address are packed, the workspace holds what the
    plan stores there, and every stream-K schedule covers each (tile,
    k-block) exactly once."""
    import random
    rng = random.Random(4242)
    seen = {}
    for _ in range(500):
        dt = rng.choice([(DT_BF16, DT_BF16, DT_BF16), (DT_F16, DT_F16, DT_F32),
                         (DT_BF16, DT_BF16, DT_F32), TF32])
        es = 4 if dt[0] == DT_F32 else 2
        M = rng.choice([rng.randint(1, 64), rng.randint(65, 512), rng.randint(513, 6000)])
        N = rng.choice([rng.randint(1, 256), rng.randint(257, 8192)])
        K = rng.choice([rng.randint(1, 128), rng.randint(129, 8192)])
        ta, tb = rng.choice("NT"), rng.choice("NT")
        rows_a, cols_a = (M, K) if ta == "N" else (K, M)
        rows_b, cols_b = (K, N) if tb == "N" else (N, K)
        lda = cols_a + rng.choice([0, 0, (-cols_a) % 8, 1])
        ldb = cols_b + rng.choice([0, 0, (-cols_b) % 8, 3])
        ldc = N + rng.choice([0, (-N) % 8])
        pa = 256 + rng.choice([0, 0, es])
        sms = rng.choice([152, 148, 132, 7])
        beta = rng.choice([0.0, 1.0])
        st, p = lib.gemm_plan_query(ta, tb, M, N, K, 1.0, pa, lda, 256, ldb, beta, 256, ldc, dt,
                                    num_sms=sms)
        assert st == 0, (ta, tb, M, N, K, lda, ldb, ldc, dt)
        path = p["path_name"]
        seen[path] = seen.get(path, 0) + 1
        if path not in ("tiled_1sm", "tiled_2sm", "skinny"):
            continue
        Mk, Nk = (N, M) if p["swap_ab"] else (M, N)
        assert p["tiles_m"] == -(-Mk // p["block_m"]) and p["tiles_n"] == -(-Nk // p["block_n"])
        assert p["num_tiles"] == p["tiles_m"] * p["tiles_n"]
        assert 1 <= p["grid"] <= sms and (path != "tiled_2sm" or p["grid"] % 2 == 0)
        assert p["k_blocks"] == -(-K // p["block_k"])
        # TMA needs 16-byte row pitches and bases: otherwise the operand is packed
        # (FP32 operands stored M/N-contiguous are transposed instead)
        a_ok = (lda * es) % 16 == 0 and pa % 16 == 0
        b_ok = (ldb * es) % 16 == 0
        if not a_ok:
            assert p["pack_a"] or p["transpose_ab"] or p["swap_ab"] and p["pack_b"], p
        if not b_ok:
            assert p["pack_b"] or p["transpose_ab"] or p["swap_ab"] and p["pack_a"], p
        if p["sk_len"] > 0:
            simulate_stream_k(p)
        else:
            assert p["sk_max_seg"] == 0 or p["sk_len"] == 0
    assert seen.get("tiled_2sm", 0) > 20 and seen.get("tiled_1sm", 0) > 20 and seen.get("skinny", 0) > 10, seen

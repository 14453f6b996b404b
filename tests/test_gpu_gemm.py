"""Q4_K / Q6_K x Q8_K GEMM on the GPU vs the CPU oracle.

Tolerance (per element): |Y_gpu - Y_oracle| <= 2e-5 * sum_b |c_b| + 1e-6, with
c_b the oracle's fp64 per-superblock contribution.  The Q8_K operand the GEMM
consumes is the GPU quantizer's, first checked bit-exact against the oracle's.

Coverage: the benchmark workloads (full output where the oracle finishes in
seconds, seeded row samples plus every tail row at the large sizes), ragged
M / N edges around every tile size, every tile width and split-K factor,
degenerate blocks (d = 0, dmin = 0, all-zero quants, extreme sub-scales),
guard canaries around Y, the launch counters and the device status word.
"""
import contextlib

import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import (assert_q8k_equal, device_status_clean, ensure_built, gpu_gemm, gpu_quantize,
                        q8k_numpy, to_dev)
from parity_util import assert_gemm_close, oracle_gemm, sample_rows, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    # the tile GEMM for every M here (the streaming path for M <= 8 has its
    # own tests in test_gpu_smallm.py)
    ensure_built()
    small = qg.qgemm_get_option(qg.QGEMM_OPT_SMALL_M_MAX)
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 0)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, 0)
    yield
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, small)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, 0)


# Q4_K side words: made by their own kernel and loaded (threshold 0 token
# tiles), or made inside the GEMM (threshold above any tile count)
SIDE_MODES = {"side_kernel": 0, "side_in_gemm": 1 << 30}


@contextlib.contextmanager
def side_mode(mode):
    old = qg.qgemm_get_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES)
    qg.qgemm_set_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES, SIDE_MODES[mode])
    try:
        yield
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES, old)


def weights(wtype, N, K, seed):
    return (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, seed)


def check(wtype, w, K, x, rows=None, what=""):
    q = gpu_quantize(x)
    q8 = q8k_numpy(q)
    assert_q8k_equal(q8, oracle.get().quantize_q8k(x), what)
    y = gpu_gemm(wtype, w, K, q)
    yr, absc = oracle_gemm(wtype, w, K, *q8, rows=rows)
    ysel = y if rows is None else y[rows]
    return assert_gemm_close(ysel, yr, absc, what)


RAGGED = [(1, 128, 256), (2, 136, 512), (3, 1, 256), (5, 200, 768), (7, 128, 1024), (8, 256, 512),
          (9, 130, 512), (15, 128, 256), (16, 128, 512), (17, 300, 512), (31, 129, 256), (33, 128, 768),
          (63, 256, 512), (64, 128, 512), (65, 136, 512), (80, 128, 1024), (127, 128, 256),
          (128, 256, 512), (129, 130, 768), (200, 384, 512), (257, 256, 1024)]


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_shapes(wtype, M, N, K):
    w = weights(wtype, N, K, 31 + M * 7 + N)
    x = synth.gen_x(M, K, 17 + M, outlier_frac=0.01)
    check(wtype, w, K, x, what=f"Q{wtype}_K M{M} N{N} K{K}")


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("bm", [16, 32, 64, 128])
@pytest.mark.parametrize("splits", [1, 2, 3, 8])
def test_every_tile_and_split(wtype, bm, splits):
    M, N, K = 100, 300, 2048
    w = weights(wtype, N, K, 5)
    x = synth.gen_x(M, K, 6)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, bm)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, splits)
    try:
        qg.qgemm_reset_counters()
        check(wtype, w, K, x, what=f"bm{bm} splits{splits}")
        c = qg.qgemm_get_counters()
        assert c["q4k_tc" if wtype == 4 else "q6k_tc"] == 1
        assert c["split_k"] == (1 if splits > 1 else 0)
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, 0)


@pytest.mark.parametrize("wtype", [4, 6])
def test_short_last_round_is_cut(wtype):
    # more tiles than SMs, the last round 8 tiles: those are cut into K parts
    # (the planner's choice on any SM count), the rest stay whole
    G = torch.cuda.get_device_properties(0).multi_processor_count
    M, K = 200, 2048
    N = 128 * ((G + 8 + 1) // 2)                 # 2 token tiles x N/128 weight tiles = G + 8 or G + 9
    w = weights(wtype, N, K, 41)
    x = synth.gen_x(M, K, 42, outlier_frac=0.01)
    qg.qgemm_reset_counters()
    rows = np.unique(np.concatenate([sample_rows(M, 24, seed=3), [0, 127, 128, M - 1]]))
    check(wtype, w, K, x, rows=rows, what=f"Q{wtype}_K M{M} N{N} K{K} on {G} SMs")
    c = qg.qgemm_get_counters()
    assert c["q4k_tc" if wtype == 4 else "q6k_tc"] == 1 and c["split_k"] == 1, c


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M,N,K", [(1100, 300, 16384), (4096, 1280, 5120)])
def test_grouped_work_order(wtype, M, N, K):
    """fp16 activations beyond 32 MiB: token tiles are taken in groups of
    about 32 MiB (M=1100, K=16384: groups of 8 and 1 token tiles, every tile
    cut into K parts; M=4096, K=5120: groups of 24 and 8, whole tiles and a
    cut last round).  Every token tile is checked."""
    assert M * K * 2 > 32 << 20
    w = weights(wtype, N, K, 90 + M)
    x = synth.gen_x(M, K, 91 + M, outlier_frac=0.01)
    check(wtype, w, K, x, rows=tile_rows(M, 128, seed=M), what=f"grouped order Q{wtype}_K M{M} N{N} K{K}")
    device_status_clean()


def check_bench_path(wl, rows=None):
    """The workload through the call the benchmark times (fp32 X in, one call:
    qgemm_q4k_f32 / qgemm_q6k_f32 with a caller workspace), with its Q8_K
    planes bit-exact and Y (all rows, or the sampled ones) within tolerance."""
    x = wl.x()
    M, N, K = wl.M, wl.N, wl.K
    w_np = wl.weights()
    w = to_dev(w_np)
    q = qg.Q8K.empty(M, K, "cuda")
    ws = torch.empty(max(qg.qgemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device="cuda")
    xd = to_dev(x)
    if wl.wtype == 4:
        y = qg.qgemm_q4k_f32(w, N, K, xd, out=q, workspace=ws)
    else:
        y = qg.qgemm_q6k_f32(qg.qgemm_q6k_prepack(w, N, K), N, K, xd, out=q, workspace=ws)
    torch.cuda.synchronize()
    q8 = q8k_numpy(q)
    assert_q8k_equal(q8, oracle.get().quantize_q8k(x), wl.name)
    yr, absc = oracle_gemm(wl.wtype, w_np, K, *q8, rows=rows)
    yg = y.cpu().numpy()
    assert_gemm_close(yg if rows is None else yg[rows], yr, absc, wl.name)
    device_status_clean()


@pytest.mark.parametrize("wl", [synth.C0, synth.C1, synth.C2, synth.F2], ids=lambda w: w.name)
def test_workload_full(wl):
    check_bench_path(wl)


@pytest.mark.parametrize("wl", [synth.C3] + [synth.sweep(m) for m in synth.SWEEP_M],
                         ids=lambda w: w.name)
def test_workload_sampled(wl):
    # at least 256 rows, one in every 128-token tile, and the tail rows
    rows = None if wl.M <= 256 else tile_rows(wl.M, 256, seed=wl.M)
    check_bench_path(wl, rows)


def _q4k_blocks(orc, N, nb, rng, d_bits=None, dmin_bits=None, q_zero=False):
    rows = []
    for n in range(N):
        blks = []
        for b in range(nb):
            db = int(rng.integers(0x0C00, 0x1400)) if d_bits is None else d_bits
            mb = int(rng.integers(0x0C00, 0x1400)) if dmin_bits is None else dmin_bits
            q = np.zeros(256, int) if q_zero else rng.integers(0, 16, 256)
            blks.append(orc.q4k_pack(db, mb, rng.integers(0, 64, 8), rng.integers(0, 64, 8), q))
        rows.append(np.concatenate(blks))
    return np.stack(rows)


@pytest.mark.parametrize("mode", list(SIDE_MODES))
@pytest.mark.parametrize("case", ["d_zero", "dmin_zero", "both_zero", "q_zero", "max_fields"])
def test_q4k_degenerate_blocks(case, mode):
    orc = oracle.get()
    rng = np.random.default_rng(3)
    N, K, M = 130, 512, 20
    if case == "d_zero":
        w = _q4k_blocks(orc, N, 2, rng, d_bits=0)
    elif case == "dmin_zero":
        w = _q4k_blocks(orc, N, 2, rng, dmin_bits=0)
    elif case == "both_zero":
        w = _q4k_blocks(orc, N, 2, rng, d_bits=0, dmin_bits=0)
    elif case == "q_zero":
        w = _q4k_blocks(orc, N, 2, rng, q_zero=True)
    else:
        blk = orc.q4k_pack(0x3C00, 0x3C00, np.full(8, 63), np.full(8, 63), np.full(256, 15))
        w = np.tile(blk, (N, 2))
    x = synth.gen_x(M, K, 8)
    x[3] = 0.0                                        # an all-zero token row
    x[4, :256] = 127.0                                # saturated superblock
    with side_mode(mode):
        check(4, w, K, x, what=f"{case}, {mode}")
    device_status_clean()


def test_q6k_scale_edges():
    orc = oracle.get()
    rng = np.random.default_rng(4)
    N, K, M = 136, 512, 33
    rows = []
    for n in range(N):
        sc = rng.choice([-64, -63, 64, 63, 0, 1, -1, 32, -32], 16)
        blks = [orc.q6k_pack(0x3C00 if n % 3 else 0, sc, rng.integers(0, 64, 256)) for _ in range(2)]
        rows.append(np.concatenate(blks))
    w = np.stack(rows)
    check(6, w, K, synth.gen_x(M, K, 9), what="q6k sc=+-64")
    device_status_clean()


Q6K_EXTREMES = np.array([-128, -127, -65, -64, 63, 64, 65, 127])


def _q6k_full_range(orc, N, nb, seed):
    """Q6_K rows whose int8 sub-scales cover the whole range: the extremes
    (-128, -127, +-65, +-64, 63, 127) in every position, and random int8."""
    r = np.random.default_rng(seed)
    rows = []
    for n in range(N):
        blks = []
        for b in range(nb):
            if (n + b) % 3 == 0:
                sc = np.roll(Q6K_EXTREMES, n + b)[np.arange(16) % 8]
            else:
                sc = r.integers(-128, 128, 16)
            d_bits = int(r.integers(0x0C00, 0x1400))        # fp16 in [2^-12, 2^-10)
            blks.append(orc.q6k_pack(d_bits, sc, r.integers(0, 64, 256)))
        rows.append(np.concatenate(blks))
    return np.stack(rows)


@pytest.mark.parametrize("M,N,K,bm,splits", [(100, 300, 2048, 128, 1), (100, 300, 2048, 64, 2), (40, 136, 1024, 32, 3),
                                             (9, 130, 512, 16, 1), (200, 384, 2560, 0, 0), (1, 256, 768, 0, 0)])
def test_q6k_full_int8_scales(M, N, K, bm, splits):
    """Every int8 sub-scale is computed, not flagged: the tile path splits a
    sub-scale beyond +-64 into two exact fp16 parts."""
    w = _q6k_full_range(oracle.get(), N, K // 256, seed=M + N + K)
    x = synth.gen_x(M, K, 11 + M, outlier_frac=0.01)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, bm)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, splits)
    try:
        qg.qgemm_reset_counters()
        check(6, w, K, x, what=f"Q6_K full int8 scales M{M} N{N} K{K} bm{bm} splits{splits}")
        c = qg.qgemm_get_counters()
        assert c["q6k_tc"] == 1, c
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, 0)
    device_status_clean()


def test_q6k_full_int8_scales_cut_last_round():
    G = torch.cuda.get_device_properties(0).multi_processor_count
    M, K = 200, 2048
    N = 128 * ((G + 8 + 1) // 2)
    w = _q6k_full_range(oracle.get(), N, K // 256, seed=77)
    x = synth.gen_x(M, K, 78)
    qg.qgemm_reset_counters()
    rows = np.unique(np.concatenate([sample_rows(M, 24, seed=5), [0, 127, 128, M - 1]]))
    check(6, w, K, x, rows=rows, what=f"Q6_K full int8 scales, cut last round, N{N}")
    assert qg.qgemm_get_counters()["split_k"] == 1
    device_status_clean()


@pytest.mark.parametrize("mode", list(SIDE_MODES))
def test_q4k_large_dmin_ratio_is_exact(mode):
    """Blocks with |dmin/d| from 1e3 up to about 1.6e7 run on a power-of-two
    shifted scale and stay within the tolerance, with no status bit."""
    orc = oracle.get()
    r = np.random.default_rng(6)
    N, K, M = 136, 2048, 24
    rows = []
    for n in range(N):
        blks = []
        for b in range(K // 256):
            d_bits = int(r.choice([0x0001, 0x0003, 0x0100, 0x0400, 0x0800, 0x1000, 0x1400]))   # 6e-8 .. 1e-3
            dmin_bits = int(r.choice([0x3C00, 0x3800, 0x2E00, 0x2400]))                         # 1.0 .. 0.0156
            blks.append(orc.q4k_pack(d_bits, dmin_bits, r.integers(0, 64, 8), r.integers(0, 64, 8),
                                     r.integers(0, 16, 256)))
        rows.append(np.concatenate(blks))
    w = np.stack(rows)
    with side_mode(mode):
        check(4, w, K, synth.gen_x(M, K, 7), what=f"Q4_K large dmin/d, {mode}")
    device_status_clean()


@pytest.mark.parametrize("mode", list(SIDE_MODES))
def test_q4k_out_of_range_row_is_declined(mode):
    """A block whose correction leaves fp16's range even on the largest
    shifted scale is not computed: its row of Y is NaN and the status bit is
    set; every other row is exact."""
    orc = oracle.get()
    rng = np.random.default_rng(5)
    N, K, M = 128, 512, 16
    w = synth.gen_q4k(N, K, 9)
    bad_row = 37
    mn = np.full(8, 63)
    w[bad_row, :144] = orc.q4k_pack(0x0001, 0x4400, rng.integers(0, 64, 8), mn, rng.integers(0, 16, 256))  # d 6e-8, dmin 4
    q = gpu_quantize(synth.gen_x(M, K, 1))
    with side_mode(mode):
        y = gpu_gemm(4, w, K, q)
    bits, _ = qg.qgemm_get_device_status()
    assert bits & qg.QGEMM_DEV_Q4K_RANGE
    assert np.isnan(y[:, bad_row]).all()
    keep = np.arange(N) != bad_row
    yr, absc = oracle_gemm(4, w, K, *q8k_numpy(q))
    assert_gemm_close(y[:, keep], yr[:, keep], absc[:, keep], "rows beside the declined one")
    device_status_clean()


@pytest.mark.parametrize("M,N,K,bm,splits", [(64, 300, 2048, 0, 0), (100, 136, 1024, 32, 3), (128, 260, 768, 128, 1),
                                             (129, 1000, 2048, 0, 0), (300, 200, 4096, 64, 2), (520, 384, 512, 0, 0)])
def test_q4k_side_paths_agree(M, N, K, bm, splits):
    """The side words made by their own kernel and loaded, or made inside the
    GEMM: bit-equal Y, both within the oracle's tolerance, and the launch
    counters show which ran."""
    w = weights(4, N, K, 3 * M + N)
    x = synth.gen_x(M, K, 5 * M + K, outlier_frac=0.01)
    q = gpu_quantize(x)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, bm)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, splits)
    ys = {}
    try:
        for mode in SIDE_MODES:
            with side_mode(mode):
                qg.qgemm_reset_counters()
                ys[mode] = gpu_gemm(4, w, K, q)
                c = qg.qgemm_get_counters()
            assert c["q4k_tc"] == 1 and c["q4k_side"] == (1 if mode == "side_kernel" else 0), (mode, c)
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, 0)
    assert np.array_equal(ys["side_kernel"], ys["side_in_gemm"], equal_nan=True)
    yr, absc = oracle_gemm(4, w, K, *q8k_numpy(q))
    assert_gemm_close(ys["side_in_gemm"], yr, absc, f"M{M} N{N} K{K} bm{bm} splits{splits}")
    device_status_clean()


def test_q4k_side_default_threshold():
    """Default: up to three token tiles per weight tile make the side words in
    the GEMM, four or more load them from their own kernel (fp32 entry point
    and Q8_K entry point alike)."""
    assert qg.qgemm_get_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES) == 4
    N, K = 256, 1024
    w_np = weights(4, N, K, 90)
    w = to_dev(w_np)
    for M, expect in [(100, 0), (129, 0), (384, 0), (385, 1), (700, 1)]:
        x = synth.gen_x(M, K, 91 + M)
        q = gpu_quantize(x)
        qg.qgemm_reset_counters()
        y1 = gpu_gemm(4, w_np, K, q)
        c = qg.qgemm_get_counters()
        assert c["q4k_side"] == expect, (M, c)
        ws = torch.empty(qg.qgemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        qg.qgemm_reset_counters()
        y2 = qg.qgemm_q4k_f32(w, N, K, to_dev(x), workspace=ws)
        torch.cuda.synchronize()
        c = qg.qgemm_get_counters()
        assert c["q4k_side"] == expect and c["quantize"] == 1 and c["q4k_tc"] == 1, (M, c)
        assert np.array_equal(y1, y2.cpu().numpy(), equal_nan=True), M
    device_status_clean()


@pytest.mark.parametrize("wtype", [4, 6])
def test_output_canaries_and_row_stride(wtype):
    M, N, K = 70, 200, 768
    w = weights(wtype, N, K, 12)
    x = synth.gen_x(M, K, 13)
    q = gpu_quantize(x)
    ldy = N + 24
    sentinel = -1234.5
    big = torch.full((M + 2, ldy), sentinel, dtype=torch.float32, device="cuda")
    y = big[1:M + 1, :N]
    gpu_gemm(wtype, w, K, q, y=y)
    b = big.cpu().numpy()
    assert np.all(b[0] == sentinel) and np.all(b[M + 1] == sentinel), "rows outside Y touched"
    assert np.all(b[1:M + 1, N:] == sentinel), "padding columns touched"
    yr, absc = oracle_gemm(wtype, w, K, *q8k_numpy(q))
    assert_gemm_close(b[1:M + 1, :N], yr, absc, "strided Y")


def test_empty_m_is_a_noop():
    w = to_dev(weights(4, 128, 256, 1))
    q = qg.Q8K.empty(0, 256)
    y = torch.empty((0, 128), dtype=torch.float32, device="cuda")
    qg.qgemm_reset_counters()
    qg.qgemm_q4k(w, 128, 256, q, y=y)
    assert qg.qgemm_get_counters()["q4k_tc"] == 0


def test_bad_workspace_is_rejected():
    w = to_dev(weights(4, 128, 512, 1))
    q = gpu_quantize(synth.gen_x(8, 512, 2))
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(qg.QgemmError) as ei:
        qg.qgemm_q4k(w, 128, 512, q, workspace=small)
    assert ei.value.code == qg.QGEMM_EINVAL


def test_device_status_clean_at_end():
    device_status_clean()

"""The small-M streaming path (M <= 8 tokens) on the GPU vs the CPU oracle.

Same tolerance as the tile GEMM: |Y_gpu - Y_oracle| <= 2e-5 * sum_b |c_b| +
1e-6.  The path is selected with QGEMM_OPT_SMALL_M_MAX; the launch counters
prove which kernel ran.  Coverage: every token count 1..8, ragged N, K from
one superblock to the path's limit, padded weight rows, degenerate blocks,
Q6_K sub-scales beyond the tensor path's fp16 range, guard canaries, the
fall-back to the tile GEMM above the K limit, and the default routing.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import assert_q8k_equal, device_status_clean, ensure_built, gpu_gemm, gpu_quantize, q8k_numpy, to_dev
from parity_util import assert_gemm_close, oracle_gemm

pytestmark = pytest.mark.gpu

K_LIMIT = 15360   # 15 consumer warps x 4 superblocks x 256


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    old = qg.qgemm_get_option(qg.QGEMM_OPT_SMALL_M_MAX)
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 8)
    yield
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, old)


def weights(wtype, N, K, seed):
    return (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, seed)


def run_small(wtype, w, K, x, what, expect_small=True, ldy_pad=0):
    q = gpu_quantize(x)
    q8 = q8k_numpy(q)
    assert_q8k_equal(q8, oracle.get().quantize_q8k(x), what)
    qg.qgemm_reset_counters()
    y = gpu_gemm(wtype, w, K, q, ldy_pad=ldy_pad)
    c = qg.qgemm_get_counters()
    small, tc = ("q4k_small", "q4k_tc") if wtype == 4 else ("q6k_small", "q6k_tc")
    if expect_small:
        assert (c[small], c[tc], c["xprep"]) == (1, 0, 0), f"{what}: counters {c}"
    else:
        assert (c[small], c[tc]) == (0, 1), f"{what}: counters {c}"
    yr, absc = oracle_gemm(wtype, w, K, *q8)
    assert_gemm_close(y, yr, absc, what)
    return y


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_token_count(wtype, M):
    N, K = 300, 2048
    run_small(wtype, weights(wtype, N, K, 100 + M), K, synth.gen_x(M, K, 200 + M, outlier_frac=0.01),
              f"Q{wtype}_K M{M}")


SHAPES = [(1, 1, 256), (2, 7, 256), (8, 1, 512), (3, 129, 768), (8, 130, 1024), (4, 33, 1280),
          (8, 64, 2560), (6, 257, 4096), (8, 200, 5120), (5, 40, 11008), (8, 24, K_LIMIT)]


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shapes(wtype, M, N, K):
    run_small(wtype, weights(wtype, N, K, 7 * N + K), K, synth.gen_x(M, K, N + M), f"Q{wtype}_K M{M} N{N} K{K}")


# Each CTA streams more stages than its shared-memory ring holds, so the
# producer waits for consumed slots and refills them.  Ring geometry for these
# launches on 152 SMs (stages per CTA against ring slots): Q4_K M=1 K=1024,
# 12 against 5; Q6_K M=8 K=2048, 20 against 8; Q4_K M=5 K=5120, 27 against 11.
@pytest.mark.parametrize("wtype,M,N,K", [(4, 1, 96000, 1024), (6, 8, 40000, 2048), (4, 5, 24000, 5120)])
def test_ring_wraps(wtype, M, N, K):
    run_small(wtype, weights(wtype, N, K, 3 * M + 1), K, synth.gen_x(M, K, 5 * M + 2, outlier_frac=0.01),
              f"Q{wtype}_K M{M} N{N} K{K} (ring wraps)")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_sweep_workload(M):
    wl = synth.sweep(M)
    run_small(wl.wtype, wl.weights(), wl.K, wl.x(), wl.name)


def test_padded_weight_rows():
    M, N, K = 5, 70, 1024
    w = weights(4, N, K, 3)
    pad = 48   # row stride 624 B: a multiple of 16 above the 576 B of blocks
    wp = np.zeros((N, w.shape[1] + pad), np.uint8)
    wp[:, : w.shape[1]] = w
    x = synth.gen_x(M, K, 4)
    q = gpu_quantize(x)
    q8 = q8k_numpy(q)
    y = torch.full((M, N), float("nan"), device="cuda")
    qg.qgemm_reset_counters()
    qg.qgemm_q4k(to_dev(wp), N, K, q, y=y)   # the row stride comes from the tensor
    torch.cuda.synchronize()
    assert qg.qgemm_get_counters()["q4k_small"] == 1
    yr, absc = oracle_gemm(4, w, K, *q8)
    assert_gemm_close(y.cpu().numpy(), yr, absc, "padded rows")


def _degenerate_q4k(orc, N, nb, rng, case):
    rows = []
    for n in range(N):
        blks = []
        for b in range(nb):
            db = 0 if case in ("d_zero", "both_zero") else int(rng.integers(0x0C00, 0x1400))
            mb = 0 if case in ("dmin_zero", "both_zero") else int(rng.integers(0x0C00, 0x1400))
            if case == "max_fields":
                db, mb = 0x7BFF, 0x7BFF   # largest finite fp16
                sc, mn, q = np.full(8, 63), np.full(8, 63), np.full(256, 15)
            else:
                sc, mn, q = rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)
            blks.append(orc.q4k_pack(db, mb, sc, mn, q))
        rows.append(np.concatenate(blks))
    return np.stack(rows)


@pytest.mark.parametrize("case", ["d_zero", "dmin_zero", "both_zero", "max_fields"])
def test_q4k_degenerate_blocks(case):
    orc = oracle.get()
    rng = np.random.default_rng(11)
    M, N, K = 3, 40, 768
    w = _degenerate_q4k(orc, N, K // 256, rng, case)
    x = synth.gen_x(M, K, 12)
    if case == "max_fields":
        x = x * 1e-3   # keep |Y| finite in fp32
    run_small(4, w, K, x, case)


def test_q6k_full_scale_range():
    """The streaming path has no fp16 operand: sub-scales -128..127 are exact."""
    orc = oracle.get()
    rng = np.random.default_rng(13)
    M, N, K = 8, 33, 1024
    rows = []
    for n in range(N):
        blks = []
        for b in range(K // 256):
            sc = rng.integers(-128, 128, 16)
            sc[0], sc[1] = -128, 127
            blks.append(orc.q6k_pack(int(rng.integers(0x0C00, 0x1400)), sc, rng.integers(0, 64, 256)))
        rows.append(np.concatenate(blks))
    w = np.stack(rows)
    run_small(6, w, K, synth.gen_x(M, K, 14), "q6k sc -128..127")
    bits, _ = qg.qgemm_get_device_status()
    assert bits == 0


@pytest.mark.parametrize("wtype", [4, 6])
def test_canaries_and_row_stride(wtype):
    M, N, K = 7, 100, 512
    run_small(wtype, weights(wtype, N, K, 21), K, synth.gen_x(M, K, 22), "ldy pad", ldy_pad=13)
    # the pad columns of Y must be untouched
    x = synth.gen_x(M, K, 22)
    q = gpu_quantize(x)
    y_full = torch.full((M, N + 13), 12345.0, device="cuda")
    gpu_gemm(wtype, weights(wtype, N, K, 21), K, q, y=y_full[:, :N])
    assert torch.all(y_full[:, N:] == 12345.0)


def test_above_k_limit_uses_tile_path():
    M, N, K = 4, 130, K_LIMIT + 256
    run_small(4, weights(4, N, K, 5), K, synth.gen_x(M, K, 6), "K over the limit", expect_small=False)


def test_default_routing():
    """Library default: M <= 8 takes the streaming path, M = 9 the tile GEMM."""
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, qg.QGEMM_SMALL_M_DEFAULT)
    try:
        N, K = 130, 1024
        w = weights(4, N, K, 41)
        run_small(4, w, K, synth.gen_x(8, K, 42), "default M8", expect_small=True)
        run_small(4, w, K, synth.gen_x(9, K, 43), "default M9", expect_small=False)
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 8)


def test_device_status_clean_at_end():
    device_status_clean()

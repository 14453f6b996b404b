"""PTQ1_0 ternary weights (qgemm_ptq1_prepack / qgemm_ptq1) on the GPU vs the
CPU oracle's codec and GEMM: |Y - Y_oracle| <= 2e-5 * sum_b |c_b| + 1e-6.

Coverage: the repack's bytes, ragged M / N around every tile width, every
tile width forced, cut tiles, a sampled K = 5120 workload (the pages measure
PTQ1_0 on K = 5120 projections), blocks with d = 0 and all-extreme trits, the
launch counters and the device status."""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import assert_q8k_equal, device_status_clean, ensure_built, gpu_quantize, q8k_numpy, to_dev
from parity_util import assert_gemm_close, oracle_gemm, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
    yield
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)


def run(w_np, K, q):
    N = w_np.shape[0]
    wp = qg.qgemm_ptq1_prepack(to_dev(w_np), N, K)
    y = qg.qgemm_ptq1(wp, N, K, q)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check(w, K, x, rows=None, what=""):
    q = gpu_quantize(x)
    qg.qgemm_reset_counters()
    y = run(w, K, q)
    c = qg.qgemm_get_counters()
    assert c["ptq1_tc"] == 1 and c["ptq1_prepack"] == 1, c
    yr, absc = oracle_gemm(1, w, K, *q8k_numpy(q), rows=rows)
    assert_gemm_close(y if rows is None else y[rows], yr, absc, what)


def test_prepack_bytes():
    N, K = 5, 768
    w = synth.gen_ptq1(N, K, 3)
    wp = qg.qgemm_ptq1_prepack(to_dev(w), N, K).cpu().numpy()
    blocks = w.reshape(N, K // 128, 28)
    want = np.concatenate([blocks, np.zeros((N, K // 128, 4), np.uint8)], axis=2).reshape(N, K // 4)
    assert np.array_equal(wp, want)


@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (3, 130, 512), (9, 200, 768), (17, 128, 1024), (64, 256, 512),
                                   (65, 136, 512), (128, 256, 1024), (129, 130, 768), (257, 384, 512)])
def test_ragged_shapes(M, N, K):
    check(synth.gen_ptq1(N, K, 11 + M), K, synth.gen_x(M, K, 12 + M, outlier_frac=0.01), what=f"M{M} N{N} K{K}")


@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_every_tile_width(bm):
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, bm)
    try:
        check(synth.gen_ptq1(300, 2048, 21), 2048, synth.gen_x(100, 2048, 22), what=f"bm{bm}")
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)


def test_extreme_blocks():
    orc = oracle.get()
    N, K, M = 128, 512, 40
    r = np.random.default_rng(7)
    blocks = []
    for n in range(N):
        row = []
        for b in range(K // 128):
            kind = (n + b) % 4
            t = (np.full(128, 2) if kind == 0 else np.zeros(128, int) if kind == 1
                 else r.integers(0, 3, 128))
            d_bits = 0x0000 if kind == 3 else int(r.integers(0x1400, 0x2400))
            row.append(orc.ptq1_pack(d_bits, t))
        blocks.append(np.concatenate(row))
    check(np.stack(blocks), K, synth.gen_x(M, K, 8), what="extreme PTQ1_0 blocks")


def test_k5120_sampled():
    M, N, K = 512, 5120, 5120
    check(synth.gen_ptq1(N, K, 31), K, synth.gen_x(M, K, 32), rows=tile_rows(M, 256, seed=4), what="M512 K5120 N5120")


def test_prepared_workspace():
    M, N, K = 70, 260, 1024
    w = synth.gen_ptq1(N, K, 41)
    x = synth.gen_x(M, K, 42)
    wp = qg.qgemm_ptq1_prepack(to_dev(w), N, K)
    ws = torch.empty(qg.qgemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    q = qg.qgemm_quantize_q8k_prep(to_dev(x), ws)
    y = qg.qgemm_ptq1_prepared(wp, N, K, q, ws)
    torch.cuda.synchronize()
    yr, absc = oracle_gemm(1, w, K, *q8k_numpy(q))
    assert_gemm_close(y.cpu().numpy(), yr, absc, "PTQ1_0 prepared")


@pytest.mark.parametrize("M,N,K", [(1, 130, 512), (70, 260, 1024), (2048, 5120, 5120)])
def test_fp32_in(M, N, K):
    """qgemm_ptq1_f32 (fp32 X in, one call, the call the benchmark times):
    the Q8_K planes bit-exact, Y within tolerance (sampled rows at the
    benchmark's 2048 x 5120 x 5120)."""
    w = synth.gen_ptq1(N, K, 51 + M)
    x = synth.gen_x(M, K, 52 + M, outlier_frac=0.01)
    wp = qg.qgemm_ptq1_prepack(to_dev(w), N, K)
    q = qg.Q8K.empty(M, K, "cuda")
    qg.qgemm_reset_counters()
    y = qg.qgemm_ptq1_f32(wp, N, K, to_dev(x), out=q)
    torch.cuda.synchronize()
    c = qg.qgemm_get_counters()
    assert (c["quantize"], c["ptq1_tc"], c["xprep"]) == (1, 1, 0), c
    q8 = q8k_numpy(q)
    assert_q8k_equal(q8, oracle.get().quantize_q8k(x), f"PTQ1_0 fp32 in M{M}")
    rows = None if M <= 256 else tile_rows(M, 256, seed=M)
    yr, absc = oracle_gemm(1, w, K, *q8, rows=rows)
    yg = y.cpu().numpy()
    assert_gemm_close(yg if rows is None else yg[rows], yr, absc, f"PTQ1_0 fp32 in M{M} N{N} K{K}")


def test_device_status_clean_at_end():
    device_status_clean()

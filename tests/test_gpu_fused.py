"""fp32 activations in, Y out (qgemm_q4k_f32 / qgemm_q6k_f32) on the GPU vs the
CPU oracle.

For M <= 2 on the small-M path the weight-streaming kernel quantizes the
activations itself; its Q8_K planes must be the oracle's bit for bit, and Y
must match the oracle's GEMM of those planes within the GEMM tolerance
(|Y_gpu - Y_oracle| <= 2e-5 * sum_b |c_b| + 1e-6).  Larger M take the
quantizer and then the small-M or tile GEMM; the launch counters show which
path ran.  Coverage: every block count pattern of the small kernel's lanes
(one superblock, partly filled warps, the K limit), ragged N, a row stride,
pinned host X, adversarial rows (ties, subnormal and underflowing scales,
zero and huge values) and near-tie rows of the quantizer's shortcut.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import assert_q8k_equal, device_status_clean, ensure_built, q8k_numpy, to_dev
from oracle_pins import _adversarial_rows
from parity_util import assert_gemm_close, oracle_gemm
from test_gpu_quantize import _near_tie_rows

pytestmark = pytest.mark.gpu

K_LIMIT = 15360


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    old = qg.qgemm_get_option(qg.QGEMM_OPT_SMALL_M_MAX)
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 8)
    yield
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, old)


def weights(wtype, N, K, seed):
    return (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, seed)


def run_f32(wtype, w_np, K, x_t, what, ldy_pad=0):
    """Y and the Q8_K planes from the fp32 entry point; checks both against
    the oracle and returns the launch counters."""
    N = w_np.shape[0]
    M = x_t.shape[0]
    w = to_dev(w_np)
    y = torch.full((M, N + ldy_pad), 7.0, dtype=torch.float32, device="cuda")
    q = qg.Q8K.empty(M, K, "cuda")
    ws = torch.empty(max(qg.qgemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device="cuda")
    qg.qgemm_reset_counters()
    if wtype == 4:
        qg.qgemm_q4k_f32(w, N, K, x_t, out=q, y=y[:, :N], workspace=ws)
    else:
        wp = qg.qgemm_q6k_prepack(w, N, K)
        qg.qgemm_reset_counters()
        qg.qgemm_q6k_f32(wp, N, K, x_t, out=q, y=y[:, :N], workspace=ws)
    torch.cuda.synchronize()
    c = qg.qgemm_get_counters()
    x_np = x_t.cpu().numpy()
    q8 = q8k_numpy(q)
    assert_q8k_equal(q8, oracle.get().quantize_q8k(np.ascontiguousarray(x_np)), what + " (Q8_K planes)")
    yr, absc = oracle_gemm(wtype, w_np, K, *q8)
    yg = y.cpu().numpy()
    assert_gemm_close(yg[:, :N], yr, absc, what)
    if ldy_pad:
        assert np.all(yg[:, N:] == 7.0), f"{what}: padding columns written"
    device_status_clean()
    return c


def expect_path(c, wtype, M, what):
    small, tc = ("q4k_small", "q4k_tc") if wtype == 4 else ("q6k_small", "q6k_tc")
    if M <= 2:
        assert (c["small_fused"], c[small], c["quantize"], c[tc]) == (1, 1, 0, 0), f"{what}: counters {c}"
    elif M <= 8:
        assert (c["small_fused"], c[small], c["quantize"], c[tc]) == (0, 1, 1, 0), f"{what}: counters {c}"
    else:
        assert (c["small_fused"], c[small], c["quantize"], c[tc]) == (0, 0, 1, 1), f"{what}: counters {c}"


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 64])
def test_every_path(wtype, M):
    N, K = 300, 2048
    x = to_dev(synth.gen_x(M, K, 300 + M, outlier_frac=0.01))
    what = f"Q{wtype}_K M{M} fp32 in"
    expect_path(run_f32(wtype, weights(wtype, N, K, 40 + M), K, x, what), wtype, M, what)


# one superblock (a quarter-filled warp); 21 superblocks (a warp with one of
# its four blocks); the small path's K limit; ragged N throughout
SHAPES = [(1, 1, 256), (2, 7, 256), (1, 129, 768), (2, 33, 5376), (1, 200, 5120), (2, 40, 11008), (1, 24, K_LIMIT),
          (2, 5, K_LIMIT)]


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_shapes(wtype, M, N, K):
    x = to_dev(synth.gen_x(M, K, 11 * N + M, outlier_frac=0.01))
    what = f"Q{wtype}_K M{M} N{N} K{K} fused"
    expect_path(run_f32(wtype, weights(wtype, N, K, 3 * N + K), K, x, what, ldy_pad=3), wtype, M, what)


@pytest.mark.parametrize("wtype", [4, 6])
def test_fused_adversarial_rows(wtype):
    """Ties, subnormal x, subnormal and underflowing scales, zero and huge
    values, two rows per call (the fused kernel's largest M)."""
    rows = _adversarial_rows(1024)
    ties = np.zeros((1, 1024), np.float32)
    ties[0, :12] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, -127.0, 3.5, -3.5, 0.49999997, -0.49999997]
    big = np.full((1, 1024), 3.0e38, np.float32)
    big[0, ::3] *= -1
    x = np.concatenate([rows, ties, big])
    N = 70
    w_np = weights(wtype, N, 1024, 17)
    for i in range(0, x.shape[0], 2):
        xs = x[i:i + 2]
        if np.abs(xs).max() > 1e30:
            # Y overflows for these rows; the Q8_K planes are what is checked
            q = qg.Q8K.empty(xs.shape[0], 1024, "cuda")
            w = to_dev(w_np)
            if wtype == 4:
                qg.qgemm_q4k_f32(w, N, 1024, to_dev(xs), out=q)
            else:
                qg.qgemm_q6k_f32(qg.qgemm_q6k_prepack(w, N, 1024), N, 1024, to_dev(xs), out=q)
            torch.cuda.synchronize()
            assert_q8k_equal(q8k_numpy(q), oracle.get().quantize_q8k(xs), f"adversarial rows {i}, {i + 1}")
            continue
        run_f32(wtype, w_np, 1024, to_dev(xs), f"Q{wtype}_K adversarial rows {i}, {i + 1}")


@pytest.mark.parametrize("M", [1, 2, 5, 40])
def test_q6k_full_int8_scales(M):
    """Q6_K sub-scales over the whole int8 range (real quantizers use it),
    on the fused, small-M and tile paths."""
    N, K = 150, 2560
    w_np = synth.gen_q6k(N, K, 61 + M, full_scales=True)
    x = to_dev(synth.gen_x(M, K, 62 + M, outlier_frac=0.01))
    what = f"Q6_K full int8 scales M{M}"
    expect_path(run_f32(6, w_np, K, x, what), 6, M, what)


def test_tile_path_ragged():
    """The tile path through the fp32 entry point on ragged M and N (several
    token and weight tiles, cut tiles)."""
    M, N, K = 300, 1000, 4096
    x = to_dev(synth.gen_x(M, K, 71, outlier_frac=0.01))
    what = "Q4_K M300 N1000 K4096 fp32 in"
    expect_path(run_f32(4, weights(4, N, K, 72), K, x, what, ldy_pad=5), 4, M, what)


def test_fused_near_ties():
    """Values on or one or two ulps beside rounding boundaries: the fused
    kernel's reciprocal shortcut must hand them to the exact division."""
    x = _near_tie_rows(K=2048, seed=21)
    w_np = weights(4, 50, 2048, 23)
    for i in range(0, 4, 2):
        run_f32(4, w_np, 2048, to_dev(x[i:i + 2]), f"near-tie rows {i}, {i + 1}")


def test_fused_row_stride_and_host_x():
    M, K, N = 2, 1280, 77
    x = synth.gen_x(M, K, 5, outlier_frac=0.01)
    wide = np.zeros((M, K + 64), np.float32)
    wide[:, :K] = x
    w_np = weights(4, N, K, 9)
    c = run_f32(4, w_np, K, to_dev(wide)[:, :K], "ldx = K + 64")
    expect_path(c, 4, M, "ldx = K + 64")
    xh = torch.from_numpy(x).pin_memory()
    c = run_f32(4, w_np, K, xh, "pinned host X")
    expect_path(c, 4, M, "pinned host X")


def test_fused_equals_two_calls():
    """Bit-equal Y from the one-launch path and from quantize + GEMM."""
    M, N, K = 2, 1000, 4096
    x = to_dev(synth.gen_x(M, K, 77, outlier_frac=0.01))
    w = to_dev(weights(4, N, K, 78))
    y1 = qg.qgemm_q4k_f32(w, N, K, x)
    q = qg.qgemm_quantize_q8k(x)
    y2 = qg.qgemm_q4k(w, N, K, q)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)

"""Tile GEMM with several work items per CTA, vs the CPU oracle.

Each persistent CTA walks tiles blockIdx.x, blockIdx.x + #SMs, ... .  At every
tile boundary, the finished tile is stored through TMEM and the accumulator of
the tile's last superblock is released to the MMA only after that store.
These cases give every CTA two or more tiles, so those hand-offs are all
exercised:
- token tiles of 128 and 64 rows;
- a ragged last token tile and a ragged last weight tile;
- a short last round cut into K parts;
- the output epilogue (bias, activation, fp16 / bf16 output).

The oracle computes sampled token rows in full (every weight tile).  Each
sampled row therefore covers every tile boundary of the launch.
Tolerance: |Y - Y_oracle| <= 2e-5 * sum_b |c_b| + 1e-6; with an output
epilogue, plus the output type's rounding as in test_gpu_epilogue.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import device_status_clean, ensure_built, gpu_quantize, q8k_numpy, to_dev
from parity_util import assert_gemm_close, oracle_gemm, tile_rows

pytestmark = pytest.mark.gpu

OUT = {"f32": (torch.float32, 0.0), "f16": (torch.float16, 2.0 ** -11), "bf16": (torch.bfloat16, 2.0 ** -8)}
ACT = {"none": qg.QGEMM_ACT_NONE, "silu": qg.QGEMM_ACT_SILU, "gelu": qg.QGEMM_ACT_GELU}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    small = qg.qgemm_get_option(qg.QGEMM_OPT_SMALL_M_MAX)
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 0)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_SPLITS, 0)
    yield
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, small)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def tiles(M, N, bm):
    return ((M + bm - 1) // bm) * ((N + 127) // 128)


def run(wtype, w_np, K, q, out=None, bias=None, act=qg.QGEMM_ACT_NONE):
    N = w_np.shape[0]
    w = to_dev(w_np)
    if wtype == 6:
        w = qg.qgemm_q6k_prepack(w, N, K)
    qg.qgemm_reset_counters()
    if out is None:
        y = qg.qgemm_q4k(w, N, K, q) if wtype == 4 else qg.qgemm_q6k(w, N, K, q)
    else:
        b = None if bias is None else to_dev(bias)
        f = qg.qgemm_q4k_ex if wtype == 4 else qg.qgemm_q6k_ex
        y = f(w, N, K, q, out_dtype=out, bias=b, activation=act)
    torch.cuda.synchronize()
    assert qg.qgemm_get_counters()["q4k_tc" if wtype == 4 else "q6k_tc"] == 1
    return y.float().cpu().numpy().astype(np.float64)


# (M, N, K, token tile): more tiles than SMs (152 on GB300), ragged edges, and
# in the last two rows a short last round cut into K parts (K = 2048: 172
# tiles, the last 20 in 4 parts; 462 tiles, the last 6 in 4 parts)
SHAPES = [(300, 15400, 512, 128), (100, 20480, 512, 64), (200, 11008, 2048, 128), (130, 19712, 2048, 64)]


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M,N,K,bm", SHAPES)
def test_several_tiles_per_cta(wtype, M, N, K, bm):
    assert tiles(M, N, bm) > sm_count()
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, bm)
    try:
        w = (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, 50 + M)
        x = synth.gen_x(M, K, 51 + M, outlier_frac=0.01)
        q = gpu_quantize(x)
        y = run(wtype, w, K, q)
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
    rows = tile_rows(M, 32, 52 + M, bm=bm, tail=3)
    yr, absc = oracle_gemm(wtype, w, K, *q8k_numpy(q), rows=rows)
    assert_gemm_close(y[rows], yr, absc, f"Q{wtype}_K M{M} N{N} K{K} BM{bm}")
    device_status_clean()


@pytest.mark.parametrize("out_name,act_name", [("f16", "silu"), ("bf16", "gelu"), ("f32", "none")])
@pytest.mark.parametrize("bm", [128, 64])
def test_several_tiles_per_cta_with_epilogue(out_name, act_name, bm):
    M, N, K = (150, 25600, 256) if bm == 128 else (90, 20480, 512)
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, bm)
    try:
        w = synth.gen_q4k(N, K, 61)
        x = synth.gen_x(M, K, 62, outlier_frac=0.01)
        bias = (synth.normal(63, N) * 0.5).astype(np.float32)
        q = gpu_quantize(x)
        out, rel = OUT[out_name]
        y = run(4, w, K, q, out=out, bias=bias, act=ACT[act_name])
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
    rows = tile_rows(M, 32, 64, bm=bm, tail=3)
    yr, absc = oracle_gemm(4, w, K, *q8k_numpy(q), rows=rows)
    ref = oracle.get().epilogue(yr, bias, ACT[act_name])
    tol = 1.2 * (2e-5 * absc + 1e-6) + (5e-6 + rel) * np.abs(ref) + 1e-6
    err = np.abs(y[rows] - ref)
    bad = err > tol
    assert not bad.any(), f"{out_name} {act_name} BM{bm}: {bad.sum()} elements, max err {err.max():.3g}"
    device_status_clean()

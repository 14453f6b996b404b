"""The GEMM with its output epilogue (qgemm_q4k_ex / qgemm_q6k_ex: output type
fp32 / fp16 / bf16, optional bias, ReLU / SiLU / GELU) on the GPU vs the
oracle's fp64 GEMM followed by the oracle's fp64 epilogue.

Tolerance per element: the GEMM bound scaled by 1.2 (each activation's slope
is at most ~1.13), plus 5e-6 |ref| for the fp32 activation (SiLU uses the fast
exponential and divide: a few 1e-6 relative), plus the output type's half-ulp
(2^-11 |ref| for fp16, 2^-8 |ref| for bf16), plus 1e-6."""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import device_status_clean, ensure_built, gpu_quantize, q8k_numpy, to_dev
from parity_util import oracle_gemm

pytestmark = pytest.mark.gpu

OUT = {"f32": (torch.float32, 0.0), "f16": (torch.float16, 2.0 ** -11), "bf16": (torch.bfloat16, 2.0 ** -8)}
ACT = {"none": qg.QGEMM_ACT_NONE, "relu": qg.QGEMM_ACT_RELU, "silu": qg.QGEMM_ACT_SILU, "gelu": qg.QGEMM_ACT_GELU}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield


def run_ex(wtype, w_np, K, q, out, bias, act):
    N = w_np.shape[0]
    w = to_dev(w_np)
    b = None if bias is None else to_dev(bias)
    if wtype == 4:
        y = qg.qgemm_q4k_ex(w, N, K, q, out_dtype=out, bias=b, activation=act)
    else:
        y = qg.qgemm_q6k_ex(qg.qgemm_q6k_prepack(w, N, K), N, K, q, out_dtype=out, bias=b, activation=act)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


def check(wtype, M, N, K, out_name, act_name, with_bias, seed):
    w = (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, seed)
    x = synth.gen_x(M, K, seed + 1, outlier_frac=0.01)
    bias = (synth.normal(seed + 2, N) * 0.5).astype(np.float32) if with_bias else None
    q = gpu_quantize(x)
    out, rel = OUT[out_name]
    y = run_ex(wtype, w, K, q, out, bias, ACT[act_name])
    yr, absc = oracle_gemm(wtype, w, K, *q8k_numpy(q))
    ref = oracle.get().epilogue(yr, bias, ACT[act_name])
    tol = 1.2 * (2e-5 * absc + 1e-6) + (5e-6 + rel) * np.abs(ref) + 1e-6
    err = np.abs(y - ref)
    bad = err > tol
    assert not bad.any(), (f"Q{wtype}_K M{M} {out_name} {act_name} bias={with_bias}: {bad.sum()} elements, "
                           f"max err {err.max():.3g}")


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("out_name", sorted(OUT))
@pytest.mark.parametrize("act_name", sorted(ACT))
def test_tile_path(wtype, out_name, act_name):
    check(wtype, 70, 260, 1024, out_name, act_name, True, seed=11 + wtype)


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("out_name", sorted(OUT))
@pytest.mark.parametrize("act_name", ["none", "gelu"])
def test_tile_path_many_token_tiles(wtype, out_name, act_name):
    # five token tiles per weight tile: Q4_K loads the side words made by
    # their own kernel (QGEMM_OPT_Q4K_SIDE_MIN_TILES, default 4)
    check(wtype, 520, 260, 1024, out_name, act_name, True, seed=51 + wtype)


@pytest.mark.parametrize("out_name", sorted(OUT))
@pytest.mark.parametrize("act_name", ["none", "relu"])
def test_tile_path_narrow_token_tile(out_name, act_name):
    # M = 20: 32-token tiles, whose store goes from registers (not through TMEM)
    check(4, 20, 260, 1024, out_name, act_name, True, seed=61)


@pytest.mark.parametrize("M", [70, 520])
@pytest.mark.parametrize("out_name,act_name,with_bias", [("f32", "none", True), ("bf16", "none", False),
                                                         ("f16", "silu", True), ("bf16", "gelu", True)])
def test_q4k_side_forms_agree(M, out_name, act_name, with_bias):
    """The epilogue GEMM with the Q4_K side words from their own kernel or made
    in the GEMM: bit-equal output, and the launch counters show which ran."""
    K, N = 1024, 260
    w = to_dev(synth.gen_q4k(N, K, 71 + M))
    q = gpu_quantize(synth.gen_x(M, K, 72 + M, outlier_frac=0.01))
    b = to_dev((synth.normal(73, N) * 0.5).astype(np.float32)) if with_bias else None
    out = OUT[out_name][0]
    old = qg.qgemm_get_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES)
    ys = []
    try:
        for mode in (0, 1 << 30):
            qg.qgemm_set_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES, mode)
            qg.qgemm_reset_counters()
            ys.append(qg.qgemm_q4k_ex(w, N, K, q, out_dtype=out, bias=b, activation=ACT[act_name]))
            torch.cuda.synchronize()
            c = qg.qgemm_get_counters()
            assert c["q4k_tc"] == 1 and c["q4k_side"] == (1 if mode == 0 else 0), (mode, c)
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES, old)
    assert torch.equal(ys[0], ys[1])
    device_status_clean()


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("out_name", sorted(OUT))
@pytest.mark.parametrize("act_name", ["none", "silu"])
def test_small_m_path(wtype, out_name, act_name):
    check(wtype, 5, 200, 1024, out_name, act_name, True, seed=21 + wtype)


@pytest.mark.parametrize("out_name", sorted(OUT))
def test_no_bias_and_cut_tiles(out_name):
    # 3 weight tiles over the SMs: cut into K parts, the epilogue after the fix-up
    check(4, 100, 300, 2048, out_name, "gelu", False, seed=31)


def test_default_epilogue_is_the_plain_gemm():
    K, N, M = 1024, 300, 90
    w = synth.gen_q4k(N, K, 41)
    q = gpu_quantize(synth.gen_x(M, K, 42))
    wd = to_dev(w)
    y0 = qg.qgemm_q4k(wd, N, K, q)
    y1 = qg.qgemm_q4k_ex(wd, N, K, q)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)


def test_device_status_clean_at_end():
    device_status_clean()

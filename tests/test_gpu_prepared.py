"""Quantize-and-prepare (qgemm_quantize_q8k_prep) and the prepared GEMMs on the
GPU: the Q8_K planes stay bit-exact with the oracle, the operand planes the
quantizer writes into the workspace are byte-identical to what the separate
preparation launch writes, and Y through the prepared calls matches the
oracle (same tolerance as the other GEMM tests) with one launch fewer."""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import assert_q8k_equal, device_status_clean, ensure_built, q8k_numpy, to_dev
from parity_util import assert_gemm_close, oracle_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield


def _plane_views(ws: torch.Tensor, M: int, K: int):
    a = lambda n: (n + 255) // 256 * 256
    Mp = (M + 3) // 4 * 4
    o1 = a(M * K * 2)
    o2 = o1 + a(M * (K // 16) * 2)
    return ws[: M * K * 2], ws[o1: o1 + M * (K // 16) * 2], ws[o2: o2 + (K // 256) * Mp * 4]


@pytest.mark.parametrize("M,K", [(1, 256), (3, 512), (9, 768), (62, 1024), (100, 2048), (257, 512)])
def test_workspace_planes_match_the_preparation_launch(M, K):
    x = synth.gen_x(M, K, 70 + M, outlier_frac=0.01)
    xd = to_dev(x)
    N = 130
    w = to_dev(synth.gen_q4k(N, K, 71))
    need = qg.qgemm_workspace_bytes(M, N, K)
    ws_a = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    ws_b = torch.full((need,), 0xCD, dtype=torch.uint8, device="cuda")
    qa = qg.qgemm_quantize_q8k_prep(xd, ws_a)
    # reference planes: the plain GEMM call runs the separate preparation into ws_b
    old = qg.qgemm_get_option(qg.QGEMM_OPT_SMALL_M_MAX)
    qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 0)
    try:
        qb = qg.qgemm_quantize_q8k(xd)
        qg.qgemm_q4k(w, N, K, qb, workspace=ws_b)
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, old)
    torch.cuda.synchronize()
    assert_q8k_equal(q8k_numpy(qa), q8k_numpy(qb), "prep vs plain quantizer")
    for pa, pb, what in zip(_plane_views(ws_a, M, K), _plane_views(ws_b, M, K), ("xh", "xbs", "dxT")):
        assert torch.equal(pa, pb), f"M{M} K{K}: {what} plane differs"


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("M,N,K", [(1, 128, 512), (8, 200, 1024), (9, 130, 768), (65, 136, 512),
                                   (128, 256, 1024), (200, 384, 2048)])
def test_prepared_gemm_vs_oracle(wtype, M, N, K):
    x = synth.gen_x(M, K, 80 + M)
    wn = (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, 81 + N)
    w = to_dev(wn)
    if wtype == 6:
        w = qg.qgemm_q6k_prepack(w, N, K)
    ws = torch.empty(max(qg.qgemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device="cuda")
    qg.qgemm_reset_counters()
    q = qg.qgemm_quantize_q8k_prep(to_dev(x), ws)
    y = (qg.qgemm_q4k_prepared if wtype == 4 else qg.qgemm_q6k_prepared)(w, N, K, q, ws)
    torch.cuda.synchronize()
    c = qg.qgemm_get_counters()
    small = M <= qg.qgemm_get_option(qg.QGEMM_OPT_SMALL_M_MAX)
    tc, sm = ("q4k_tc", "q4k_small") if wtype == 4 else ("q6k_tc", "q6k_small")
    assert (c["quantize"], c["xprep"], c[tc], c[sm]) == (1, 0, 0 if small else 1, 1 if small else 0), c
    q8 = q8k_numpy(q)
    assert_q8k_equal(q8, oracle.get().quantize_q8k(x), "prep quantizer")
    yr, absc = oracle_gemm(wtype, wn, K, *q8)
    assert_gemm_close(y.cpu().numpy(), yr, absc, f"prepared Q{wtype}_K M{M} N{N} K{K}")


def test_benchmark_workload_prepared():
    wl = synth.C1
    x, wn = wl.x(), wl.weights()
    ws = torch.empty(qg.qgemm_workspace_bytes(wl.M, wl.N, wl.K), dtype=torch.uint8, device="cuda")
    q = qg.qgemm_quantize_q8k_prep(to_dev(x), ws)
    y = qg.qgemm_q4k_prepared(to_dev(wn), wl.N, wl.K, q, ws)
    torch.cuda.synchronize()
    yr, absc = oracle_gemm(4, wn, wl.K, *q8k_numpy(q))
    assert_gemm_close(y.cpu().numpy(), yr, absc, wl.name)


def test_device_status_clean_at_end():
    device_status_clean()

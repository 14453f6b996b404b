"""X, expert ids and Y in page-locked host memory (zero-copy): the quantizer
reads X and the GEMMs write Y across the host link themselves.

Every case runs twice on the same inputs, once with device buffers and once
with pinned host buffers, and the two results must be bit-identical (the
kernels and their reduction order are the same; only where the bytes live
differs).  One case per path is also held to the oracle: Q8_K bit-exact, Y
within |Y - Y_oracle| <= 2e-5 * sum_b |c_b| + 1e-6.

Paths: quantizer (plain and with the operand planes), tile GEMM with cut
tiles, small-M streaming kernel, fused epilogue (fp16 output), expert-routed
GEMM (ids and Y on the host), PTQ1_0."""
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
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
    yield


def pinned(a) -> torch.Tensor:
    t = a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory()


def pinned_empty(shape, dtype=torch.float32) -> torch.Tensor:
    return torch.full(shape, float("nan") if dtype.is_floating_point else 0, dtype=dtype).pin_memory()


def same_bits(a: torch.Tensor, b: torch.Tensor, what: str):
    a, b = a.cpu().contiguous(), b.cpu().contiguous()
    assert a.shape == b.shape and a.dtype == b.dtype, what
    ia = a.view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.view(torch.int16 if b.element_size() == 2 else torch.int32)
    bad = (ia != ib).nonzero()
    assert bad.numel() == 0, f"{what}: {bad.shape[0]} elements differ, first {bad[:3].tolist()}"


@pytest.mark.parametrize("M,K", [(37, 512), (300, 2048)])
def test_quantizer_reads_host_x(M, K):
    x = synth.gen_x(M, K, 11 + M, outlier_frac=0.01)
    qd = qg.qgemm_quantize_q8k(to_dev(x))
    qh = qg.qgemm_quantize_q8k(pinned(x))
    torch.cuda.synchronize()
    assert qh.qs.is_cuda      # the planes stay on the device
    assert_q8k_equal(q8k_numpy(qh), q8k_numpy(qd), "host X vs device X")
    assert_q8k_equal(q8k_numpy(qh), oracle.get().quantize_q8k(x), "host X vs oracle")
    device_status_clean()


@pytest.mark.parametrize("wtype", [4, 6])
def test_tile_gemm_prepared_host_x_and_y(wtype):
    # 5 x 3 tiles of 128 x 128 at BM 128 leave a short last round: cut tiles included
    M, N, K = 300, 520, 1024
    w_np = (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, 21 + wtype)
    x = synth.gen_x(M, K, 22, outlier_frac=0.01)
    w = to_dev(w_np)
    if wtype == 6:
        w = qg.qgemm_q6k_prepack(w, N, K)
    mm = qg.qgemm_q4k_prepared if wtype == 4 else qg.qgemm_q6k_prepared

    def run(xin, y):
        ws = torch.empty(max(qg.qgemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device="cuda")
        q = qg.qgemm_quantize_q8k_prep(xin, ws)
        mm(w, N, K, q, ws, y=y)
        torch.cuda.synchronize()
        return q, y

    _, yd = run(to_dev(x), torch.empty((M, N), device="cuda"))
    qh, yh = run(pinned(x), pinned_empty((M, N)))
    same_bits(yh, yd, f"Q{wtype}_K host Y vs device Y")
    yr, absc = oracle_gemm(wtype, w_np, K, *q8k_numpy(qh))
    assert_gemm_close(yh.numpy(), yr, absc, f"Q{wtype}_K host Y vs oracle")
    device_status_clean()


def test_tile_gemm_host_y_with_row_stride():
    M, N, K = 130, 256, 512
    w_np = synth.gen_q4k(N, K, 31)
    q = qg.qgemm_quantize_q8k(to_dev(synth.gen_x(M, K, 32)))
    w = to_dev(w_np)
    yd = qg.qgemm_q4k(w, N, K, q)
    big = pinned_empty((M, N + 40))
    yh = big[:, :N]
    qg.qgemm_q4k(w, N, K, q, y=yh)
    torch.cuda.synchronize()
    same_bits(yh, yd, "strided host Y")
    assert torch.isnan(big[:, N:]).all(), "columns past N were written"


@pytest.mark.parametrize("M", [1, 5, 8])
def test_small_m_host_y(M):
    N, K = 1000, 2048
    w_np = synth.gen_q4k(N, K, 41 + M)
    q = qg.qgemm_quantize_q8k(pinned(synth.gen_x(M, K, 42 + M)))
    w = to_dev(w_np)
    qg.qgemm_reset_counters()
    yd = qg.qgemm_q4k(w, N, K, q)
    yh = qg.qgemm_q4k(w, N, K, q, y=pinned_empty((M, N)))
    torch.cuda.synchronize()
    assert qg.qgemm_get_counters()["q4k_small"] == 2
    same_bits(yh, yd, f"small-M M={M} host Y")
    yr, absc = oracle_gemm(4, w_np, K, *q8k_numpy(q))
    assert_gemm_close(yh.numpy(), yr, absc, f"small-M M={M} host Y vs oracle")


@pytest.mark.parametrize("M", [4, 200])
def test_epilogue_fp16_host_y(M):
    N, K = 384, 1024
    w_np = synth.gen_q4k(N, K, 51)
    q = qg.qgemm_quantize_q8k(to_dev(synth.gen_x(M, K, 52)))
    w = to_dev(w_np)
    bias = to_dev(np.random.default_rng(53).standard_normal(N).astype(np.float32))
    yd = qg.qgemm_q4k_ex(w, N, K, q, out_dtype=torch.float16, bias=bias, activation=qg.QGEMM_ACT_SILU)
    yh = qg.qgemm_q4k_ex(w, N, K, q, out_dtype=torch.float16, bias=bias, activation=qg.QGEMM_ACT_SILU,
                         y=pinned_empty((M, N), torch.float16))
    torch.cuda.synchronize()
    same_bits(yh, yd, f"fp16 SiLU epilogue M={M} host Y")


@pytest.mark.parametrize("wtype", [4, 6])
def test_routed_host_ids_and_y(wtype):
    E, N, K, M, top_k = 8, 256, 1024, 90, 2
    w_np = (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(E * N, K, 61 + wtype)
    ids_np = synth.gen_ids(M, top_k, E, 62, 1.0).astype(np.int32)
    q = qg.qgemm_quantize_q8k(to_dev(synth.gen_x(M, K, 63, outlier_frac=0.01)))
    w = to_dev(w_np)
    if wtype == 6:
        w = qg.qgemm_q6k_prepack(w, E * N, K)
    mm = qg.qgemm_q4k_id if wtype == 4 else qg.qgemm_q6k_id
    yd = mm(w, E, N, K, q, to_dev(ids_np))
    yh = mm(w, E, N, K, q, pinned(ids_np), y=pinned_empty((M * top_k, N)))
    torch.cuda.synchronize()
    same_bits(yh, yd, f"routed Q{wtype}_K host ids and Y")
    yr, absc = oracle.get().gemm_id(wtype, w_np, E, K, *q8k_numpy(q), ids_np)
    assert_gemm_close(yh.numpy(), yr, absc, f"routed Q{wtype}_K host Y vs oracle")
    device_status_clean()


def test_ptq1_host_x_and_y():
    M, N, K = 200, 384, 1280
    w_np = synth.gen_ptq1(N, K, 71)
    x = synth.gen_x(M, K, 72)
    wp = qg.qgemm_ptq1_prepack(to_dev(w_np), N, K)

    def run(xin, y):
        ws = torch.empty(max(qg.qgemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device="cuda")
        q = qg.qgemm_quantize_q8k_prep(xin, ws)
        qg.qgemm_ptq1_prepared(wp, N, K, q, ws, y=y)
        torch.cuda.synchronize()
        return y

    yd = run(to_dev(x), torch.empty((M, N), device="cuda"))
    yh = run(pinned(x), pinned_empty((M, N)))
    same_bits(yh, yd, "PTQ1_0 host X and Y")

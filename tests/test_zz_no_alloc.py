"""qgemm_q4k_noalloc: the allocation-free variant of the Q4_K GEMM.

It exists for callers that cannot allocate device memory where they call the
GEMM (a plugin whose host framework owns all device memory, or code where
cudaMalloc is not allowed); it takes its scratch from a fixed device array in
the library instead of a caller workspace.  This file is collected last so a
run that stops at the first failure has already run every other test.

Checked here, through the C ABI: three calls in a row (of different shapes, so
each runs over the previous one's leftover scratch) each match the CPU
oracle's Y within the GEMM tolerance, and give the same bits as the workspace
entry point qgemm_q4k on the same inputs; a call too large for the built-in
scratch is refused without launching anything.
"""
import ctypes

import pytest
import torch

import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import ensure_built, gpu_quantize, q8k_numpy, to_dev
from parity_util import assert_gemm_close, oracle_gemm

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 16 << 20


def _noalloc(L, w, N, K, q, y):
    return L.qgemm_q4k_noalloc(ctypes.c_void_p(w.data_ptr()), N, K, w.stride(0),
                               ctypes.c_void_p(q.qs.data_ptr()), ctypes.c_void_p(q.d.data_ptr()),
                               ctypes.c_void_p(q.bsums.data_ptr()), q.M, ctypes.c_void_p(y.data_ptr()),
                               y.stride(0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_oracle_twice():
    ensure_built()
    L = qg.lib()
    # (the third shape has five token tiles per weight tile: the Q4_K side words
    # are then made by their own kernel into the built-in scratch)
    for call, (M, N, K) in enumerate(((300, 520, 2048), (37, 256, 1024), (520, 384, 1024))):
        w_np = synth.gen_q4k(N, K, 61 + call)
        x_np = synth.gen_x(M, K, 62 + call, outlier_frac=0.01)
        w = to_dev(w_np)
        q = gpu_quantize(x_np)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(L, w, N, K, q, y)
        assert rc == qg.QGEMM_OK, L.qgemm_last_error().decode()
        torch.cuda.synchronize()
        y_or, absc = oracle_gemm(4, w_np, K, *q8k_numpy(q))
        assert_gemm_close(y.cpu().numpy(), y_or, absc, f"noalloc call {call + 1} vs the oracle")
        # the same kernels as the workspace entry point: the same bits
        qg.qgemm_reset_counters()
        y_ws = qg.qgemm_q4k(w, N, K, q)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ws), f"noalloc call {call + 1}: Y differs from qgemm_q4k's"
        assert qg.qgemm_get_counters()["q4k_side"] == (1 if M > 3 * 128 else 0)
    bits, site = qg.qgemm_get_device_status()
    assert bits == 0, f"device status {bits:#x} site {site}"


def test_noalloc_refuses_more_than_its_scratch():
    ensure_built()
    L = qg.lib()
    M, N, K = 4096, 128, 4096                          # needs ~35 MB of scratch
    assert qg.qgemm_workspace_bytes(M, N, K) > NOALLOC_SCRATCH_BYTES
    w = torch.zeros((N, (K // 256) * 144), dtype=torch.uint8, device="cuda")
    q = qg.Q8K.empty(M, K)
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    qg.qgemm_reset_counters()
    rc = _noalloc(L, w, N, K, q, y)
    assert rc == qg.QGEMM_EUNSUPPORTED
    assert b"scratch" in L.qgemm_last_error()
    assert qg.qgemm_get_counters()["q4k_tc"] == 0     # nothing launched

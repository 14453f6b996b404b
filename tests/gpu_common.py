"""Shared set-up for the GPU tests: build the library once, move data to the
device, run the library's quantizer and GEMMs through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import block_quantized_matmul_quantize_gb300 as qg
from block_quantized_matmul_quantize_gb300 import build as qbuild


def ensure_built():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    qbuild.build()
    qg.lib()


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_quantize(x_np: np.ndarray):
    q = qg.qgemm_quantize_q8k(to_dev(x_np))
    torch.cuda.synchronize()
    return q


def q8k_numpy(q: qg.Q8K):
    return q.qs.cpu().numpy(), q.d.cpu().numpy(), q.bsums.cpu().numpy()


def assert_q8k_equal(got, ref, what=""):
    qs, d, bs = got
    rqs, rd, rbs = ref
    assert np.array_equal(qs, rqs), f"{what}: int8 values differ at {np.argwhere(qs != rqs)[:5].tolist()}"
    assert np.array_equal(d.view(np.uint32), rd.view(np.uint32)), f"{what}: scales differ"
    assert np.array_equal(bs, rbs), f"{what}: bsums differ"


def gpu_gemm(wtype: int, w_np: np.ndarray, K: int, q: qg.Q8K, ldy_pad: int = 0, y=None):
    """Run the GEMM through the binding; returns the fp32 output as numpy."""
    N = w_np.shape[0]
    w = to_dev(w_np)
    M = q.M
    if y is None:
        y = torch.empty((M, N + ldy_pad), dtype=torch.float32, device="cuda")[:, :N]
    if wtype == 4:
        qg.qgemm_q4k(w, N, K, q, y=y)
    else:
        wp = qg.qgemm_q6k_prepack(w, N, K)
        qg.qgemm_q6k(wp, N, K, q, y=y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def device_status_clean():
    bits, site = qg.qgemm_get_device_status()
    assert bits == 0 and site == 0, f"device status bits={bits:#x} site={site}"

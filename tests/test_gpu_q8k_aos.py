"""Q8_K planes <-> the pages' 292-byte block ("BlockQ8_K (292B/256 elements)",
vllm.cpp PR #3036, commit 4) through the C ABI, against the oracle's
conversions (oracle_q8k_to_aos / oracle_q8k_from_aos): bit-exact in both
directions, on ragged M and several K; and the caller-owned Q8_K buffer
sized by qgemm_q8k_bytes holds the quantizer's planes."""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import assert_q8k_equal, device_status_clean, ensure_built, gpu_quantize, q8k_numpy, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(1, 256), (3, 768), (37, 2048), (130, 11008), (8, 5120)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("M,K", SHAPES)
def test_pack_matches_oracle(M, K):
    x = synth.gen_x(M, K, 700 + M, outlier_frac=0.01)
    x[0, :256] = 0.0                                  # a d = 0 superblock
    q = gpu_quantize(x)
    aos = qg.qgemm_pack_q8k_aos(q)
    torch.cuda.synchronize()
    ref = oracle.get().q8k_to_aos(*q8k_numpy(q)).reshape(-1)
    assert aos.numel() == ref.size == M * (K // 256) * 292
    got = aos.cpu().numpy()
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("M,K", SHAPES)
def test_unpack_matches_oracle(M, K):
    orc = oracle.get()
    # an AoS array made by the oracle from random field values (not from the GPU)
    r = np.random.default_rng(800 + M)
    qs = r.integers(-127, 128, (M, K)).astype(np.int8)
    d = (r.random((M, K // 256)) * 1e-2).astype(np.float32)
    bs = qs.reshape(M, K // 16, 16).astype(np.int32).sum(axis=2).astype(np.int16)
    aos = orc.q8k_to_aos(qs, d, bs).reshape(-1)
    got = qg.qgemm_unpack_q8k_aos(to_dev(aos), M, K)
    torch.cuda.synchronize()
    assert_q8k_equal(q8k_numpy(got), orc.q8k_from_aos(aos, M, K), f"unpack M{M} K{K}")
    # and back again: the same bytes
    again = qg.qgemm_pack_q8k_aos(got)
    torch.cuda.synchronize()
    assert np.array_equal(again.cpu().numpy(), aos)


def test_caller_owned_q8k_buffer():
    M, K = 33, 1280
    buf = torch.empty(qg.qgemm_q8k_bytes(M, K), dtype=torch.uint8, device="cuda")
    q = qg.q8k_in_buffer(buf, M, K)
    x = synth.gen_x(M, K, 901)
    qg.qgemm_quantize_q8k(to_dev(x), out=q)
    torch.cuda.synchronize()
    assert_q8k_equal(q8k_numpy(q), oracle.get().quantize_q8k(x), "Q8_K in one caller buffer")
    device_status_clean()

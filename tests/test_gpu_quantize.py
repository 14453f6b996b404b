"""Q8_K quantizer on the GPU vs the CPU oracle: bit-exact int8 values, fp32
scales and int16 sums, on the benchmark workloads' activations and on
adversarial rows (ties, zeros, subnormals, outliers, huge values)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import assert_q8k_equal, ensure_built, gpu_quantize, q8k_numpy, to_dev
from oracle_pins import _adversarial_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


X_WORKLOADS = [synth.C0, synth.C1, synth.C2, synth.C3] + [synth.sweep(m) for m in synth.SWEEP_M]


@pytest.mark.parametrize("wl", X_WORKLOADS, ids=lambda w: w.name)
def test_quantize_bitexact_workloads(wl):
    x = wl.x()
    got = q8k_numpy(gpu_quantize(x))
    assert_q8k_equal(got, oracle.get().quantize_q8k(x), wl.name)


def test_quantize_adversarial():
    rows = _adversarial_rows(1024)
    ties = np.zeros((1, 1024), np.float32)
    ties[0, :12] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, -127.0, 3.5, -3.5, 0.49999997, -0.49999997]
    ties[0, 256:260] = [-1e-45, 1e-45, 0.0, -0.0]       # smallest subnormals, signed zeros
    big = np.full((1, 1024), 3.0e38, np.float32)
    big[0, ::3] *= -1
    x = np.concatenate([rows, ties, big])
    got = q8k_numpy(gpu_quantize(x))
    assert_q8k_equal(got, oracle.get().quantize_q8k(x), "adversarial")


def _near_tie_rows(K=2048, seed=9):
    """Chunks whose values sit on, or one or two ulps beside, the rounding
    boundaries (k + 1/2) * d of their own scale d, over scales from 1e-30 to
    1e30: the quantizer's reciprocal shortcut must hand these to the exact
    division and agree with the oracle bit for bit."""
    r = np.random.default_rng(seed)
    rows = []
    for i in range(16):
        row = np.empty(K, np.float32)
        for c in range(K // 256):
            amax = np.float32(10.0 ** r.uniform(-30, 30)) * np.float32(r.uniform(1, 2))
            d = np.float32(amax / np.float32(127))
            k = r.integers(-127, 127, 256)
            v = ((k + 0.5) * np.float64(d)).astype(np.float32)
            step = r.integers(-2, 3, 256)
            for _ in range(2):
                v = np.where(step > 0, np.nextafter(v, np.float32(np.inf)), np.where(step < 0, np.nextafter(v, np.float32(-np.inf)), v))
                step = step - np.sign(step)
            v = np.clip(v, -amax, amax)
            v[0] = amax if i % 2 else -amax
            row[256 * c:256 * c + 256] = v
        rows.append(row)
    return np.stack(rows)


def test_quantize_near_ties():
    x = _near_tie_rows()
    assert_q8k_equal(q8k_numpy(gpu_quantize(x)), oracle.get().quantize_q8k(x), "near ties")
    # the variant that also writes the GEMM's operand planes
    M, K = x.shape
    ws = torch.empty(qg.qgemm_workspace_bytes(M, 128, K), dtype=torch.uint8, device="cuda")
    q = qg.qgemm_quantize_q8k_prep(to_dev(x), ws)
    torch.cuda.synchronize()
    assert_q8k_equal(q8k_numpy(q), oracle.get().quantize_q8k(x), "near ties, with operand planes")


def test_quantize_row_stride():
    x = synth.gen_x(37, 768, 5, outlier_frac=0.01)
    wide = np.zeros((37, 1024), np.float32)
    wide[:, :768] = x
    xd = to_dev(wide)[:, :768]
    q = qg.qgemm_quantize_q8k(xd)
    torch.cuda.synchronize()
    assert_q8k_equal(q8k_numpy(q), oracle.get().quantize_q8k(x), "ldx=1024")


def test_quantize_empty_and_counter():
    qg.qgemm_reset_counters()
    q = qg.qgemm_quantize_q8k(torch.empty((0, 512), dtype=torch.float32, device="cuda"))
    assert q.M == 0
    gpu_quantize(synth.gen_x(3, 512, 1))
    assert qg.qgemm_get_counters()["quantize"] == 1

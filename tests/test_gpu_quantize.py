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

"""The kernels' bounded waits, run out on purpose, with no GPU fault.

A test-only switch (QGEMM_OPT_TEST_SKIP_ARRIVAL) makes the first CTA of a
kernel leave out one copy, so that the waits for it find nothing; with the
wait limit set to 1 ms (QGEMM_OPT_WAIT_LIMIT_US) they give up, the CTA's
other roles stop at once, and the kernel returns.  Checked: the device status
reports the timeout and the site of the wait that gave up
(qgemm_get_device_status returns QGEMM_ETIMEOUT), that CTA's output tile is
left as it was, every other output element matches the oracle, and the
context stays usable -- the same call without the switch is then exact and
the status clean.  (The pages' convention: a failure is a status the caller
can act on, not a wrong answer or a hang; hip-ep PR #627, the launcher's
failure return.)"""
import time

import numpy as np
import pytest
import torch

import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import device_status_clean, ensure_built, gpu_gemm, gpu_quantize, q8k_numpy
from parity_util import assert_gemm_close, oracle_gemm

pytestmark = pytest.mark.gpu

SENTINEL = -7.25
# The kernels' wait sites.  In the tile GEMM every role of the first CTA
# starts waiting at once, so the first of the waits downstream of the left-out
# weight copy to pass its deadline records the site: the unpack's (7) or the
# Q4_K side-data writer's (15) wait for that copy, the MMA thread's wait for
# the operand (12), or the epilogue's waits for the accumulator (10) and the
# side data (11).  In the small-M kernel it is the consumers' wait for the
# first stage (22).
TILE_SITES = {4: (7, 10, 11, 12, 15), 6: (7, 10, 11, 12)}
SITE_SMALLM_FULL = 22


@pytest.fixture
def one_ms_waits():
    ensure_built()
    device_status_clean()
    qg.qgemm_set_option(qg.QGEMM_OPT_WAIT_LIMIT_US, 1000)
    yield
    qg.qgemm_set_option(qg.QGEMM_OPT_TEST_SKIP_ARRIVAL, 0)
    qg.qgemm_set_option(qg.QGEMM_OPT_WAIT_LIMIT_US, 0)
    qg.qgemm_get_device_status()


def _run_with_skip(wtype, w, K, q, skip, M, N):
    y = torch.full((M, N), SENTINEL, dtype=torch.float32, device="cuda")
    qg.qgemm_set_option(qg.QGEMM_OPT_TEST_SKIP_ARRIVAL, skip)
    try:
        t0 = time.time()
        out = gpu_gemm(wtype, w, K, q, y=y)          # (synchronizes)
        elapsed = time.time() - t0
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_TEST_SKIP_ARRIVAL, 0)
    rc, bits, site = qg.qgemm_device_status_code()
    return out, elapsed, rc, bits, site


@pytest.mark.parametrize("wtype", [4, 6])
def test_tile_gemm_wait_runs_out(one_ms_waits, wtype):
    # 8 weight tiles x 2 token tiles, each cut into 4 K parts: the first CTA
    # runs part 0 of tile 0 (weight rows 0..127, tokens 0..127) and nothing else
    M, N, K = 256, 1024, 2048
    w = (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, 71)
    x = synth.gen_x(M, K, 72)
    q = gpu_quantize(x)
    y, elapsed, rc, bits, site = _run_with_skip(wtype, w, K, q, 1, M, N)
    assert rc == qg.QGEMM_ETIMEOUT, rc
    assert bits & qg.QGEMM_DEV_TIMEOUT
    assert site - 1 in TILE_SITES[wtype], site
    assert elapsed < 10.0
    assert np.all(y[:128, :128] == SENTINEL), "the CTA that gave up wrote its tile"
    yr, absc = oracle_gemm(wtype, w, K, *q8k_numpy(q))
    keep = np.ones((M, N), bool)
    keep[:128, :128] = False
    assert_gemm_close(y[keep], yr[keep], absc[keep], "the tiles of the other CTAs")
    # the context is usable: the same call again, without the switch
    y2 = gpu_gemm(wtype, w, K, q)
    assert_gemm_close(y2, yr, absc, "the call after the timeout")
    device_status_clean()


def test_smallm_wait_runs_out(one_ms_waits):
    M, N, K = 4, 5120, 5120
    w = synth.gen_q4k(N, K, 73)
    x = synth.gen_x(M, K, 74)
    q = gpu_quantize(x)
    qg.qgemm_reset_counters()
    y, elapsed, rc, bits, site = _run_with_skip(4, w, K, q, 2, M, N)
    assert qg.qgemm_get_counters()["q4k_small"] == 1
    assert rc == qg.QGEMM_ETIMEOUT and bits & qg.QGEMM_DEV_TIMEOUT and site - 1 == SITE_SMALLM_FULL, (rc, bits, site)
    assert elapsed < 10.0
    grid = min(torch.cuda.get_device_properties(0).multi_processor_count, N)
    r1 = N // grid                                   # the first CTA's weight rows: 0 .. r1-1
    assert np.all(y[:, :r1] == SENTINEL), "the CTA that gave up wrote its rows"
    yr, absc = oracle_gemm(4, w, K, *q8k_numpy(q))
    assert_gemm_close(y[:, r1:], yr[:, r1:], absc[:, r1:], "the rows of the other CTAs")
    y2 = gpu_gemm(4, w, K, q)
    assert_gemm_close(y2, yr, absc, "the call after the timeout")
    device_status_clean()

"""Expert-routed GEMM (qgemm_q4k_id / qgemm_q6k_id, the pages' MUL_MAT_ID)
on the GPU vs the CPU oracle (oracle_gemm_id): every (token, slot) row within
the GEMM tolerance |Y - Y_oracle| <= 2e-5 * sum_b |c_b| + 1e-6.

Coverage: uniform and skewed routing (empty experts), one expert taking
everything, a token routed to the same expert twice, ragged N, every token
tile width, Q4_K and Q6_K, out-of-range ids (status bit, rows untouched),
the launch counters, and the device status word."""
import numpy as np
import pytest
import torch

import oracle
import synth
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import device_status_clean, ensure_built, gpu_quantize, q8k_numpy, to_dev
from parity_util import assert_gemm_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)
    yield
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)


def run_routed(wtype, w_np, E, K, q, ids_np, y=None):
    N = w_np.shape[0] // E
    w = to_dev(w_np)
    ids = to_dev(ids_np.astype(np.int32))
    if wtype == 4:
        y = qg.qgemm_q4k_id(w, E, N, K, q, ids, y=y)
    else:
        wp = qg.qgemm_q6k_prepack(w, E * N, K)
        y = qg.qgemm_q6k_id(wp, E, N, K, q, ids, y=y)
    torch.cuda.synchronize()
    return y


def check(wtype, E, N, K, M, top_k, seed, skew=0.0, ids=None, what=""):
    gen = synth.gen_q4k if wtype == 4 else synth.gen_q6k
    w = gen(E * N, K, seed)
    x = synth.gen_x(M, K, seed + 1, outlier_frac=0.01)
    if ids is None:
        ids = synth.gen_ids(M, top_k, E, seed + 2, skew)
    q = gpu_quantize(x)
    qg.qgemm_reset_counters()
    y = run_routed(wtype, w, E, K, q, ids).cpu().numpy()
    c = qg.qgemm_get_counters()
    assert c["routed"] == 1 and c["q4k_tc" if wtype == 4 else "q6k_tc"] == 1, c
    yr, absc = oracle.get().gemm_id(wtype, w, E, K, *q8k_numpy(q), ids)
    assert_gemm_close(y, yr, absc, what or f"Q{wtype}_K E{E} N{N} K{K} M{M} top{top_k}")
    return ids


@pytest.mark.parametrize("wtype", [4, 6])
@pytest.mark.parametrize("E,N,K,M,top_k", [(8, 256, 1024, 64, 2), (4, 130, 512, 33, 3), (16, 128, 512, 100, 4),
                                           (1, 384, 1024, 50, 1), (3, 200, 768, 7, 2), (32, 136, 512, 300, 2)])
def test_routed_vs_oracle(wtype, E, N, K, M, top_k):
    check(wtype, E, N, K, M, top_k, seed=100 + E * 7 + M)


@pytest.mark.parametrize("wtype", [4, 6])
def test_skewed_routing_with_empty_experts(wtype):
    ids = check(wtype, 16, 256, 1024, 200, 2, seed=31, skew=2.5)
    counts = np.bincount(ids.ravel(), minlength=16)
    assert counts.max() > 4 * counts.mean()


def test_all_tokens_to_one_expert_and_repeats():
    M, E = 150, 6
    ids = np.full((M, 2), 4, np.int32)          # both slots of every token: expert 4
    check(4, E, 256, 512, M, 2, seed=41, ids=ids)


@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_every_tile_width(bm):
    qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, bm)
    try:
        check(4, 8, 256, 1024, 90, 2, seed=51 + bm)
    finally:
        qg.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0)


def test_moe_workload_sampled():
    # a mixture-of-experts FFN projection: 8 experts, 2 per token, 256 tokens
    E, N, K, M, top_k = 8, 2816, 2048, 256, 2
    w = synth.gen_q4k(E * N, K, 61)
    x = synth.gen_x(M, K, 62)
    ids = synth.gen_ids(M, top_k, E, 63)
    q = gpu_quantize(x)
    y = run_routed(4, w, E, K, q, ids).cpu().numpy()
    tok = np.unique(np.concatenate([np.random.default_rng(5).choice(M, 12, replace=False), [0, M - 1]]))
    qs, d, bs = q8k_numpy(q)
    yr, absc = oracle.get().gemm_id(4, w, E, K, qs[tok], d[tok], bs[tok], ids[tok])
    rows = (tok[:, None] * top_k + np.arange(top_k)[None, :]).ravel()
    assert_gemm_close(y[rows], yr, absc, "moe E8 top2 M256 K2048 N2816")


def test_out_of_range_ids_flagged_rows_untouched():
    E, N, K, M = 4, 128, 512, 5
    w = synth.gen_q4k(E * N, K, 71)
    x = synth.gen_x(M, K, 72)
    ids = np.array([[0, 1], [2, -1], [3, 3], [E, 0], [1, 2]], np.int32)
    q = gpu_quantize(x)
    device_status_clean()
    y = torch.full((M * 2, N), 12345.0, dtype=torch.float32, device="cuda")
    run_routed(4, w, E, K, q, ids, y=y)
    bits, site = qg.qgemm_get_device_status()      # reads and clears
    assert bits == qg.QGEMM_DEV_BAD_EXPERT and site == 0, (bits, site)
    yn = y.cpu().numpy()
    assert (yn[3] == 12345.0).all() and (yn[6] == 12345.0).all()
    yr, absc = oracle.get().gemm_id(4, w, E, K, *q8k_numpy(q), ids)
    good = [0, 1, 2, 4, 5, 7, 8, 9]
    assert_gemm_close(yn[good], yr[good], absc[good], "valid rows beside bad ids")


def test_device_status_clean_at_end():
    device_status_clean()

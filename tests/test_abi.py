"""The C-ABI library builds, loads and exports every symbol include/qgemm.h
declares; host-side validation rejects bad arguments before touching the GPU.
No compute calls: these run without a GPU."""
import ctypes
import os
import re

import pytest

import block_quantized_matmul_quantize_gb300 as qg
from block_quantized_matmul_quantize_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qg.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qgemm_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for need in ("qgemm_quantize_q8k", "qgemm_q4k", "qgemm_q6k", "qgemm_q6k_prepack",
                 "qgemm_workspace_bytes", "qgemm_get_counters", "qgemm_get_device_status"):
        assert need in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_no_oracle_symbols_in_library(L):
    # the product library shares no code with the CPU oracle
    for n in ("oracle_gemm_q4k", "oracle_quantize_q8k", "oracle_q4k_fields"):
        with pytest.raises(AttributeError):
            getattr(L, n)


def test_version(L):
    assert L.qgemm_version() >= 100


FAKE = ctypes.c_void_p(0x100000)      # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x100004)


def test_quantize_validation(L):
    assert L.qgemm_quantize_q8k(FAKE, 1, 100, 100, FAKE, FAKE, FAKE, None) == qg.QGEMM_EINVAL
    assert b"multiple of 256" in L.qgemm_last_error()
    assert L.qgemm_quantize_q8k(FAKE, -1, 256, 256, FAKE, FAKE, FAKE, None) == qg.QGEMM_EINVAL
    assert L.qgemm_quantize_q8k(FAKE, 0, 256, 256, FAKE, FAKE, FAKE, None) == qg.QGEMM_OK   # empty
    assert L.qgemm_quantize_q8k(None, 2, 256, 256, FAKE, FAKE, FAKE, None) == qg.QGEMM_EINVAL
    assert L.qgemm_quantize_q8k(FAKE, 2, 256, 128, FAKE, FAKE, FAKE, None) == qg.QGEMM_EINVAL
    assert L.qgemm_quantize_q8k(MISALIGNED, 2, 256, 256, FAKE, FAKE, FAKE, None) == qg.QGEMM_EALIGN
    assert L.qgemm_quantize_q8k(FAKE, 2, 256, 258, FAKE, FAKE, FAKE, None) == qg.QGEMM_EALIGN
    assert L.qgemm_quantize_q8k(FAKE, 2, 256, 256, MISALIGNED, FAKE, FAKE, None) == qg.QGEMM_EALIGN
    assert L.qgemm_quantize_q8k(FAKE, 2, 256, 256, None, FAKE, FAKE, None) == qg.QGEMM_EINVAL


def test_prepared_validation(L):
    # quantize + prepare: the quantizer's checks, then the workspace's
    P = L.qgemm_quantize_q8k_prep
    assert P(FAKE, 1, 100, 100, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == qg.QGEMM_EINVAL
    assert P(FAKE, 0, 256, 256, FAKE, FAKE, FAKE, None, 0, None) == qg.QGEMM_OK       # empty
    assert P(MISALIGNED, 2, 256, 256, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == qg.QGEMM_EALIGN
    need = L.qgemm_workspace_bytes(2, 0, 256)   # N = 0: the planes and counters the quantizer writes
    assert P(FAKE, 2, 256, 256, FAKE, FAKE, FAKE, None, need, None) == qg.QGEMM_EINVAL
    assert P(FAKE, 2, 256, 256, FAKE, FAKE, FAKE, FAKE, need - 1, None) == qg.QGEMM_EINVAL
    assert P(FAKE, 2, 256, 256, FAKE, FAKE, FAKE, ctypes.c_void_p(0x100010), need, None) == qg.QGEMM_EALIGN
    # the prepared GEMMs share the plain ones' argument checks
    G = L.qgemm_q4k_prepared
    assert G(FAKE, 128, 300, 288, FAKE, FAKE, FAKE, 4, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_EINVAL
    assert G(FAKE, 128, 512, 296, FAKE, FAKE, FAKE, 4, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_EALIGN
    assert G(FAKE, 128, 512, 288, FAKE, FAKE, FAKE, 0, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_OK
    H = L.qgemm_q6k_prepared
    assert H(FAKE, 128, 384, FAKE, FAKE, FAKE, 4, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_EINVAL
    assert H(FAKE, 128, 512, FAKE, FAKE, FAKE, 4, None, 128, FAKE, 1 << 20, None) == qg.QGEMM_EINVAL


def test_gemm_validation(L):
    ws = FAKE
    args = lambda **kw: dict(dict(w=FAKE, N=128, K=512, ldw=288, qs=FAKE, d=FAKE, bs=FAKE, M=4, y=FAKE,
                                  ldy=128), **kw)

    def q4k(a):
        return L.qgemm_q4k(a["w"], a["N"], a["K"], a["ldw"], a["qs"], a["d"], a["bs"], a["M"], a["y"],
                           a["ldy"], ws, 1 << 20, None)
    assert q4k(args(K=300)) == qg.QGEMM_EINVAL
    assert q4k(args(N=0)) == qg.QGEMM_EINVAL
    assert q4k(args(M=0)) == qg.QGEMM_OK                    # empty: nothing launched
    assert q4k(args(ldw=287)) == qg.QGEMM_EINVAL           # shorter than a row of blocks
    assert q4k(args(ldw=296)) == qg.QGEMM_EALIGN           # not a multiple of 16
    assert q4k(args(w=MISALIGNED)) == qg.QGEMM_EALIGN
    assert q4k(args(w=None)) == qg.QGEMM_EINVAL
    assert q4k(args(qs=MISALIGNED)) == qg.QGEMM_EALIGN
    assert q4k(args(y=None)) == qg.QGEMM_EINVAL
    assert q4k(args(ldy=100)) == qg.QGEMM_EINVAL
    assert q4k(args(N=1 << 31)) == qg.QGEMM_EUNSUPPORTED
    assert L.qgemm_q6k(FAKE, 128, 384, FAKE, FAKE, FAKE, 4, FAKE, 128, ws, 1 << 20, None) == qg.QGEMM_EINVAL
    assert L.qgemm_q6k_prepack(FAKE, 0, 256, 210, FAKE, None) == qg.QGEMM_EINVAL
    assert L.qgemm_q6k_prepack(FAKE, 4, 256, 200, FAKE, None) == qg.QGEMM_EINVAL
    assert L.qgemm_q6k_prepack(FAKE, 4, 256, 210, MISALIGNED, None) == qg.QGEMM_EALIGN


def test_routed_validation(L):
    F, H = L.qgemm_q4k_id, L.qgemm_q6k_id
    ids_bad = ctypes.c_void_p(0x100002)

    def q4(E=8, N=128, K=512, ldw=288, M=4, ids=FAKE, top_k=2, y=FAKE, ldy=128):
        return F(FAKE, E, N, K, ldw, FAKE, FAKE, FAKE, M, ids, top_k, y, ldy, FAKE, 1 << 20, None)
    assert q4(E=0) == qg.QGEMM_EINVAL
    assert q4(E=1025) == qg.QGEMM_EINVAL
    assert q4(top_k=0) == qg.QGEMM_EINVAL
    assert q4(ids=None) == qg.QGEMM_EINVAL
    assert q4(ids=ids_bad) == qg.QGEMM_EALIGN
    assert q4(K=300) == qg.QGEMM_EINVAL
    assert q4(ldw=296) == qg.QGEMM_EALIGN
    assert q4(ldy=100) == qg.QGEMM_EINVAL
    assert q4(E=8, N=1 << 28, ldy=1 << 28) == qg.QGEMM_EUNSUPPORTED   # E * N >= 2^31
    assert q4(M=1 << 30, top_k=4) == qg.QGEMM_EUNSUPPORTED   # M * top_k >= 2^31
    assert q4(M=0) == qg.QGEMM_OK                            # empty: nothing launched
    assert H(FAKE, 8, 128, 512, FAKE, FAKE, FAKE, 4, FAKE, 0, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_EINVAL
    # routed rows: 8 pairs + 3 padding rows per expert = 32; routing 3 x 256 B + perm 32 ints (-> 256);
    # xh 32x512x2, xbs 32x32x2, dxT 2x32x4 (-> 256)
    assert L.qgemm_id_workspace_bytes(4, 2, 8, 512) == 768 + 256 + 32768 + 2048 + 256
    assert L.qgemm_id_workspace_bytes(0, 2, 8, 512) == 0
    assert L.qgemm_id_workspace_bytes(4, 0, 8, 512) == 0


def test_epilogue_validation(L):
    ep = qg._Epilogue(qg.QGEMM_OUT_F16, qg.QGEMM_ACT_SILU, None)
    F = L.qgemm_q4k_ex

    def q4(e, y=FAKE, ldy=128):
        return F(FAKE, 128, 512, 288, FAKE, FAKE, FAKE, 4, y, ldy, ctypes.byref(e) if e else None, FAKE, 1 << 20,
                 None)
    assert q4(qg._Epilogue(3, 0, None)) == qg.QGEMM_EINVAL          # unknown output type
    assert q4(qg._Epilogue(0, 4, None)) == qg.QGEMM_EINVAL          # unknown activation
    assert q4(qg._Epilogue(0, 1, 0x100002)) == qg.QGEMM_EALIGN      # bias not 4-byte aligned
    assert q4(ep, y=ctypes.c_void_p(0x100001)) == qg.QGEMM_EALIGN   # fp16 y must be 2-byte aligned
    assert q4(None, y=ctypes.c_void_p(0x100002)) == qg.QGEMM_EALIGN  # fp32 y must be 4-byte aligned
    assert q4(ep, ldy=100) == qg.QGEMM_EINVAL
    assert F(FAKE, 128, 512, 288, FAKE, FAKE, FAKE, 0, FAKE, 128, ctypes.byref(ep), FAKE, 1 << 20, None) == 0
    assert L.qgemm_q6k_ex(FAKE, 128, 384, FAKE, FAKE, FAKE, 4, FAKE, 128, ctypes.byref(ep), FAKE, 1 << 20,
                          None) == qg.QGEMM_EINVAL


def test_ptq1_validation(L):
    P, G = L.qgemm_ptq1_prepack, L.qgemm_ptq1
    assert P(FAKE, 0, 256, 56, FAKE, None) == qg.QGEMM_EINVAL
    assert P(FAKE, 4, 384, 84, FAKE, None) == qg.QGEMM_EINVAL            # K not a multiple of 256
    assert P(FAKE, 4, 256, 55, FAKE, None) == qg.QGEMM_EINVAL            # ldw < 2 blocks of 28 B
    assert P(FAKE, 4, 256, 56, MISALIGNED, None) == qg.QGEMM_EALIGN
    assert G(FAKE, 128, 300, FAKE, FAKE, FAKE, 4, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_EINVAL
    assert G(MISALIGNED, 128, 512, FAKE, FAKE, FAKE, 4, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_EALIGN
    assert G(FAKE, 128, 512, FAKE, FAKE, FAKE, 0, FAKE, 128, FAKE, 1 << 20, None) == qg.QGEMM_OK
    assert L.qgemm_ptq1_packed_bytes(3, 512) == 3 * 4 * 32
    assert L.qgemm_ptq1_packed_bytes(3, 384) == 0


def test_size_queries(L):
    assert L.qgemm_workspace_bytes(0, 8, 256) == 0
    assert L.qgemm_workspace_bytes(4, 8, 300) == 0
    M, K = 5, 512
    # xh fp16 5*512*2 = 5120; bsums fp16 5*32*2 = 320 -> 512; d^T fp32 2*8*4 = 64 -> 256
    # + the cut-tile counters (8 per tile) + the Q4_K side words (2 superblocks x 2 slabs x 8 rows x 32 B,
    # and the scales e 2 x 8 fp32 -> 256); one tile: no partial tiles
    expect = 5120 + 512 + 256 + 1024 * 8 * 4 + 1024 + 256
    assert L.qgemm_workspace_bytes(M, 8, K) == expect
    assert L.qgemm_q6k_packed_bytes(3, 512) == 3 * 2 * 224
    assert L.qgemm_q6k_packed_bytes(3, 100) == 0


def test_q8k_storage_queries(L):
    assert L.qgemm_q8k_bytes(0, 256) == 0 and L.qgemm_q8k_bytes(3, 300) == 0
    M, K = 3, 768
    # qs 2304 -> 2304 (256-B multiple), d 3*3*4 = 36 -> 256, bsums 3*48*2 = 288 -> 512
    assert L.qgemm_q8k_bytes(M, K) == 2304 + 256 + 512
    qs, d, bs = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    base = 0x100000
    assert L.qgemm_q8k_planes(ctypes.c_void_p(base), M, K, ctypes.byref(qs), ctypes.byref(d),
                              ctypes.byref(bs)) == qg.QGEMM_OK
    assert (qs.value, d.value, bs.value) == (base, base + 2304, base + 2304 + 256)
    assert L.qgemm_q8k_planes(ctypes.c_void_p(base + 16), M, K, ctypes.byref(qs), ctypes.byref(d),
                              ctypes.byref(bs)) == qg.QGEMM_EALIGN
    assert L.qgemm_q8k_planes(None, M, K, ctypes.byref(qs), ctypes.byref(d), ctypes.byref(bs)) == qg.QGEMM_EINVAL
    assert L.qgemm_q8k_planes(ctypes.c_void_p(base), M, 100, ctypes.byref(qs), ctypes.byref(d),
                              ctypes.byref(bs)) == qg.QGEMM_EINVAL
    # the pages' 292-byte block
    assert L.qgemm_q8k_aos_bytes(M, K) == M * 3 * 292
    assert L.qgemm_q8k_aos_bytes(M, 100) == 0
    P, U = L.qgemm_pack_q8k_aos, L.qgemm_unpack_q8k_aos
    assert P(FAKE, FAKE, FAKE, 0, 256, FAKE, None) == qg.QGEMM_OK            # empty
    assert P(FAKE, FAKE, FAKE, 2, 100, FAKE, None) == qg.QGEMM_EINVAL
    assert P(FAKE, FAKE, FAKE, 2, 256, None, None) == qg.QGEMM_EINVAL
    assert P(FAKE, FAKE, FAKE, 2, 256, ctypes.c_void_p(0x100002), None) == qg.QGEMM_EALIGN
    assert P(MISALIGNED, FAKE, FAKE, 2, 256, FAKE, None) == qg.QGEMM_EALIGN
    assert U(FAKE, 2, 256, FAKE, None, FAKE, None) == qg.QGEMM_EINVAL
    assert U(ctypes.c_void_p(0x100001), 2, 256, FAKE, FAKE, FAKE, None) == qg.QGEMM_EALIGN


def test_options_and_counters(L):
    assert L.qgemm_get_option(qg.QGEMM_OPT_SMALL_M_MAX) == qg.QGEMM_SMALL_M_DEFAULT == 8
    assert L.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 9) == qg.QGEMM_EINVAL
    assert L.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 0) == qg.QGEMM_OK
    assert L.qgemm_set_option(qg.QGEMM_OPT_SMALL_M_MAX, 8) == qg.QGEMM_OK
    assert L.qgemm_set_option(1, 48) == qg.QGEMM_EINVAL
    assert L.qgemm_set_option(7, 0) == qg.QGEMM_EINVAL
    assert L.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 64) == qg.QGEMM_OK
    assert L.qgemm_get_option(qg.QGEMM_OPT_FORCE_BM) == 64
    assert L.qgemm_set_option(qg.QGEMM_OPT_FORCE_BM, 0) == qg.QGEMM_OK
    assert L.qgemm_get_option(99) == -1
    # the wait limit and the test-only skip switch: range-checked before any device access
    assert L.qgemm_set_option(qg.QGEMM_OPT_WAIT_LIMIT_US, 10_000_001) == qg.QGEMM_EINVAL
    assert L.qgemm_set_option(qg.QGEMM_OPT_TEST_SKIP_ARRIVAL, 3) == qg.QGEMM_EINVAL
    assert L.qgemm_set_option(6, 0) == qg.QGEMM_EINVAL
    # the Q4_K side-data threshold: default 4 token tiles, any count up to 2^30
    assert L.qgemm_get_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES) == 4
    assert L.qgemm_set_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES, (1 << 30) + 1) == qg.QGEMM_EINVAL
    assert L.qgemm_set_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES, 0) == qg.QGEMM_OK
    assert L.qgemm_get_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES) == 0
    assert L.qgemm_set_option(qg.QGEMM_OPT_Q4K_SIDE_MIN_TILES, 4) == qg.QGEMM_OK
    L.qgemm_reset_counters()
    c = qg._Counters()
    assert L.qgemm_get_counters(ctypes.byref(c)) == 0
    assert c.q4k_tc == 0 and c.quantize == 0
    assert L.qgemm_get_counters(None) == qg.QGEMM_EINVAL


def test_binding_refuses_pageable_host_tensors(L):
    """X, ids and Y may be pinned host tensors, never pageable ones; every
    other argument must be a CUDA tensor.  The binding refuses before the
    library is called, so this runs without a GPU."""
    import torch
    out = qg.Q8K(torch.zeros((2, 256), dtype=torch.int8), torch.zeros((2, 1)),
                 torch.zeros((2, 16), dtype=torch.int16))
    with pytest.raises(ValueError, match="pinned host tensors"):
        qg.qgemm_quantize_q8k(torch.zeros((2, 256)), out=out)
    with pytest.raises(ValueError, match="CUDA tensor is required"):
        qg.qgemm_q4k(torch.zeros((8, 144), dtype=torch.uint8), 8, 256, out, y=torch.zeros((2, 8)))

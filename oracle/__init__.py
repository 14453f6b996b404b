"""CPU oracle for the k-quant prefill matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never does; the two share no code.

This module compiles ``oracle.c`` with gcc (single-threaded, no fast-math, no
FMA contraction) and wraps it with ctypes/numpy.  What the oracle computes,
and which passages it follows, is written in ``oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
DEFAULT_LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
          "-fPIC", "-shared"]

Q4K_BYTES = 144
Q6K_BYTES = 210
Q8K_BYTES = 292
PTQ1_BYTES = 28


def build(src: str = SRC, out: str = DEFAULT_LIB, force: bool = False) -> str:
    """Compile the oracle to a shared library; returns its path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(src),
                                             os.path.getmtime(os.path.join(HERE, "oracle.h")))):
        return out
    cmd = ["gcc", *CFLAGS, "-I", HERE, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes wrapper around one build of oracle.c."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = build()
        self.path = lib_path
        L = ctypes.CDLL(lib_path)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_double.restype = ctypes.c_double
        L.oracle_q4k_fields.argtypes = [vp] * 6
        L.oracle_q4k_pack.argtypes = [ctypes.c_uint16, ctypes.c_uint16, vp, vp, vp, vp]
        L.oracle_q6k_fields.argtypes = [vp] * 4
        L.oracle_q6k_pack.argtypes = [ctypes.c_uint16, vp, vp, vp]
        L.oracle_dequant_q4k.argtypes = [vp, vp]
        L.oracle_dequant_q6k.argtypes = [vp, vp]
        L.oracle_quantize_q8k.argtypes = [vp, i64, i64, i64, vp, vp, vp]
        L.oracle_q8k_to_aos.argtypes = [vp, vp, vp, i64, i64, vp]
        L.oracle_q8k_from_aos.argtypes = [vp, i64, i64, vp, vp, vp]
        L.oracle_gemm_q4k.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, vp]
        L.oracle_gemm_q6k.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, vp]
        L.oracle_brute.argtypes = [ctypes.c_int, vp, i64, i64, i64, vp, vp, i64, vp]
        L.oracle_gemm_id.argtypes = [ctypes.c_int, vp, i64, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, vp]
        L.oracle_epilogue.argtypes = [vp, i64, i64, vp, ctypes.c_int]
        L.oracle_ptq1_fields.argtypes = [vp, vp, vp]
        L.oracle_ptq1_pack.argtypes = [ctypes.c_uint16, vp, vp]
        L.oracle_dequant_ptq1.argtypes = [vp, vp]
        L.oracle_gemm_ptq1.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, i64, vp, vp]
        for f in ("oracle_q4k_fields", "oracle_q4k_pack", "oracle_q6k_fields",
                  "oracle_q6k_pack", "oracle_dequant_q4k", "oracle_dequant_q6k",
                  "oracle_quantize_q8k", "oracle_q8k_to_aos", "oracle_q8k_from_aos",
                  "oracle_gemm_q4k", "oracle_gemm_q6k", "oracle_brute"):
            getattr(L, f).restype = None
        self.L = L

    # -- formats ---------------------------------------------------------
    def half_to_double(self, bits: int) -> float:
        return self.L.oracle_half_to_double(int(bits))

    def q4k_fields(self, blk: np.ndarray):
        blk = np.ascontiguousarray(blk, dtype=np.uint8)
        d = np.zeros(1); dmin = np.zeros(1)
        sc = np.zeros(8, np.int32); mn = np.zeros(8, np.int32); q = np.zeros(256, np.int32)
        self.L.oracle_q4k_fields(_p(blk), _p(d), _p(dmin), _p(sc), _p(mn), _p(q))
        return float(d[0]), float(dmin[0]), sc, mn, q

    def q4k_pack(self, d_bits: int, dmin_bits: int, sc, mn, q) -> np.ndarray:
        sc = np.ascontiguousarray(sc, np.int32); mn = np.ascontiguousarray(mn, np.int32)
        q = np.ascontiguousarray(q, np.int32)
        blk = np.zeros(Q4K_BYTES, np.uint8)
        self.L.oracle_q4k_pack(int(d_bits), int(dmin_bits), _p(sc), _p(mn), _p(q), _p(blk))
        return blk

    def q6k_fields(self, blk: np.ndarray):
        blk = np.ascontiguousarray(blk, dtype=np.uint8)
        d = np.zeros(1); sc = np.zeros(16, np.int32); q = np.zeros(256, np.int32)
        self.L.oracle_q6k_fields(_p(blk), _p(d), _p(sc), _p(q))
        return float(d[0]), sc, q

    def q6k_pack(self, d_bits: int, sc, q) -> np.ndarray:
        sc = np.ascontiguousarray(sc, np.int32); q = np.ascontiguousarray(q, np.int32)
        blk = np.zeros(Q6K_BYTES, np.uint8)
        self.L.oracle_q6k_pack(int(d_bits), _p(sc), _p(q), _p(blk))
        return blk

    def ptq1_fields(self, blk: np.ndarray):
        """(d, t int32 [128]) of one 28-byte PTQ1_0 block (t in 0..2, value t - 1)."""
        blk = np.ascontiguousarray(blk, dtype=np.uint8)
        d = np.zeros(1); t = np.zeros(128, np.int32)
        self.L.oracle_ptq1_fields(_p(blk), _p(d), _p(t))
        return float(d[0]), t

    def ptq1_pack(self, d_bits: int, t) -> np.ndarray:
        t = np.ascontiguousarray(t, np.int32)
        blk = np.zeros(PTQ1_BYTES, np.uint8)
        self.L.oracle_ptq1_pack(int(d_bits), _p(t), _p(blk))
        return blk

    def dequant(self, wtype: int, blk: np.ndarray) -> np.ndarray:
        blk = np.ascontiguousarray(blk, dtype=np.uint8)
        if wtype == 1:
            w = np.zeros(128)
            self.L.oracle_dequant_ptq1(_p(blk), _p(w))
            return w
        w = np.zeros(256)
        fn = self.L.oracle_dequant_q4k if wtype == 4 else self.L.oracle_dequant_q6k
        fn(_p(blk), _p(w))
        return w

    # -- Q8_K --------------------------------------------------------------
    def quantize_q8k(self, x: np.ndarray):
        """x fp32 [M, K] -> (qs int8 [M,K], d fp32 [M,K/256], bsums int16 [M,K/16])."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        M, K = x.shape
        qs = np.zeros((M, K), np.int8)
        d = np.zeros((M, K // 256), np.float32)
        bs = np.zeros((M, K // 16), np.int16)
        self.L.oracle_quantize_q8k(_p(x), M, K, K, _p(qs), _p(d), _p(bs))
        return qs, d, bs

    def q8k_to_aos(self, qs, d, bs) -> np.ndarray:
        M, K = qs.shape
        out = np.zeros((M, (K // 256) * Q8K_BYTES), np.uint8)
        self.L.oracle_q8k_to_aos(_p(np.ascontiguousarray(qs)), _p(np.ascontiguousarray(d)),
                                 _p(np.ascontiguousarray(bs)), M, K, _p(out))
        return out

    def q8k_from_aos(self, aos: np.ndarray, M: int, K: int):
        aos = np.ascontiguousarray(aos, np.uint8)
        qs = np.zeros((M, K), np.int8)
        d = np.zeros((M, K // 256), np.float32)
        bs = np.zeros((M, K // 16), np.int16)
        self.L.oracle_q8k_from_aos(_p(aos), M, K, _p(qs), _p(d), _p(bs))
        return qs, d, bs

    # -- GEMM ------------------------------------------------------------
    def gemm(self, wtype: int, w: np.ndarray, K: int, qs, d, bs, rows=None):
        """w uint8 [N, nb*blockbytes]; returns (y fp64 [R, N], absc fp64 [R, N])."""
        w = np.ascontiguousarray(w, np.uint8)
        N = w.shape[0]
        qs = np.ascontiguousarray(qs, np.int8)
        d = np.ascontiguousarray(d, np.float32)
        bs = np.ascontiguousarray(bs, np.int16)
        M = qs.shape[0]
        if rows is None:
            rows_arr = np.arange(M, dtype=np.int64)
        else:
            rows_arr = np.ascontiguousarray(rows, np.int64)
            assert rows_arr.size == 0 or (rows_arr.min() >= 0 and rows_arr.max() < M)
        R = rows_arr.size
        y = np.zeros((R, N)); absc = np.zeros((R, N))
        if wtype == 1:
            self.L.oracle_gemm_ptq1(_p(w), N, K, w.shape[1], _p(qs), _p(d), M, _p(rows_arr), R, _p(y), _p(absc))
            return y, absc
        fn = self.L.oracle_gemm_q4k if wtype == 4 else self.L.oracle_gemm_q6k
        fn(_p(w), N, K, w.shape[1], _p(qs), _p(d), _p(bs), M, _p(rows_arr), R, _p(y), _p(absc))
        return y, absc

    def gemm_id(self, wtype: int, w: np.ndarray, E: int, K: int, qs, d, bs, ids):
        """w uint8 [E*N, row bytes] (E experts stacked); ids int32 [M, top_k].
        Returns (y fp64 [M*top_k, N], absc fp64 [M*top_k, N]); rows of ids outside
        [0, E) stay NaN."""
        w = np.ascontiguousarray(w, np.uint8)
        assert w.shape[0] % E == 0
        N = w.shape[0] // E
        qs = np.ascontiguousarray(qs, np.int8)
        d = np.ascontiguousarray(d, np.float32)
        bs = np.ascontiguousarray(bs, np.int16)
        ids = np.ascontiguousarray(ids, np.int32)
        M, top_k = ids.shape
        assert qs.shape[0] == M
        y = np.full((M * top_k, N), np.nan); absc = np.full((M * top_k, N), np.nan)
        self.L.oracle_gemm_id(int(wtype), _p(w), E, N, K, w.shape[1], _p(qs), _p(d), _p(bs), M, _p(ids), top_k,
                              _p(y), _p(absc))
        return y, absc

    def epilogue(self, y: np.ndarray, bias=None, act: int = 0) -> np.ndarray:
        """act(y + bias[n]) in fp64 on a copy of y [R, N] (act 0 none, 1 ReLU, 2 SiLU, 3 GELU)."""
        out = np.array(y, dtype=np.float64, order="C", copy=True)
        R, N = out.shape
        b = None if bias is None else np.ascontiguousarray(bias, np.float32)
        assert b is None or b.shape == (N,)
        self.L.oracle_epilogue(_p(out), R, N, None if b is None else _p(b), int(act))
        return out

    def brute(self, wtype: int, w: np.ndarray, K: int, qs, d) -> np.ndarray:
        w = np.ascontiguousarray(w, np.uint8)
        qs = np.ascontiguousarray(qs, np.int8)
        d = np.ascontiguousarray(d, np.float32)
        N = w.shape[0]; M = qs.shape[0]
        y = np.zeros((M, N))
        self.L.oracle_brute(int(wtype), _p(w), N, K, w.shape[1], _p(qs), _p(d), M, _p(y))
        return y


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def tolerance(absc: np.ndarray) -> np.ndarray:
    """Allowed |Y_gpu - Y_oracle| per element: 2e-5 * sum_b |c_b| + 1e-6."""
    return 2e-5 * absc + 1e-6

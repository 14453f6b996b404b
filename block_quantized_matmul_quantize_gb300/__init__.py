"""Python binding of the k-quant prefill matmul library (libqgemm.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/qgemm.h.  PyTorch provides device
memory and the current stream.  The functions carry the C names.

There is no CPU fallback: if the library has not been built, or a call fails,
a QgemmError is raised.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libqgemm.so")

QGEMM_OK, QGEMM_EINVAL, QGEMM_EALIGN, QGEMM_EUNSUPPORTED, QGEMM_ECUDA, QGEMM_ETIMEOUT, QGEMM_EDEVICE = range(7)
QGEMM_DEV_TIMEOUT, QGEMM_DEV_Q4K_RANGE, QGEMM_DEV_BAD_EXPERT = 0x1, 0x2, 0x8
QGEMM_DEBUG_EXPAND_BYTES = 1152
QGEMM_OPT_SMALL_M_MAX, QGEMM_OPT_FORCE_BM, QGEMM_OPT_FORCE_SPLITS = 0, 1, 2
QGEMM_OPT_WAIT_LIMIT_US, QGEMM_OPT_TEST_SKIP_ARRIVAL = 3, 4
QGEMM_OPT_Q4K_SIDE_MIN_TILES = 5
QGEMM_SMALL_M_DEFAULT = 8   # the library's default for QGEMM_OPT_SMALL_M_MAX

QGEMM_OUT_F32, QGEMM_OUT_F16, QGEMM_OUT_BF16 = 0, 1, 2
QGEMM_ACT_NONE, QGEMM_ACT_RELU, QGEMM_ACT_SILU, QGEMM_ACT_GELU = 0, 1, 2, 3

Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210


class QgemmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"qgemm error {code}: {msg}")
        self.code = code


class _Counters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("quantize", "xprep", "q4k_tc", "q6k_tc", "q4k_small", "q6k_small", "q6k_prepack", "split_k",
                 "routed", "ptq1_tc", "ptq1_prepack", "small_fused", "q4k_side")]


class _Epilogue(ctypes.Structure):
    _fields_ = [("out_type", ctypes.c_int), ("activation", ctypes.c_int), ("bias", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise QgemmError(QGEMM_ECUDA, f"{LIB_PATH} not found: build it first "
                             "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, sz, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
        sig = {
            "qgemm_version": ([], i32),
            "qgemm_last_error": ([], ctypes.c_char_p),
            "qgemm_quantize_q8k": ([vp, i64, i64, i64, vp, vp, vp, vp], i32),
            "qgemm_workspace_bytes": ([i64, i64, i64], sz),
            "qgemm_q8k_bytes": ([i64, i64], sz),
            "qgemm_q8k_planes": ([vp, i64, i64, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp)], i32),
            "qgemm_q8k_aos_bytes": ([i64, i64], sz),
            "qgemm_pack_q8k_aos": ([vp, vp, vp, i64, i64, vp, vp], i32),
            "qgemm_unpack_q8k_aos": ([vp, i64, i64, vp, vp, vp, vp], i32),
            "qgemm_q4k": ([vp, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_q4k_noalloc": ([vp, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp], i32),
            "qgemm_q6k_packed_bytes": ([i64, i64], sz),
            "qgemm_q6k_prepack": ([vp, i64, i64, i64, vp, vp], i32),
            "qgemm_q6k": ([vp, i64, i64, vp, vp, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_quantize_q8k_prep": ([vp, i64, i64, i64, vp, vp, vp, vp, sz, vp], i32),
            "qgemm_q4k_prepared": ([vp, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_q4k_f32": ([vp, i64, i64, i64, vp, i64, i64, vp, vp, vp, vp, i64, vp, sz, vp], i32),
            "qgemm_q6k_f32": ([vp, i64, i64, vp, i64, i64, vp, vp, vp, vp, i64, vp, sz, vp], i32),
            "qgemm_ptq1_f32": ([vp, i64, i64, vp, i64, i64, vp, vp, vp, vp, i64, vp, sz, vp], i32),
            "qgemm_q6k_prepared": ([vp, i64, i64, vp, vp, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_id_workspace_bytes": ([i64, i64, i64, i64], sz),
            "qgemm_q4k_id": ([vp, i64, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_q6k_id": ([vp, i64, i64, i64, vp, vp, vp, i64, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_q4k_ex": ([vp, i64, i64, i64, vp, vp, vp, i64, vp, i64, ctypes.POINTER(_Epilogue), vp, sz, vp],
                             i32),
            "qgemm_q6k_ex": ([vp, i64, i64, vp, vp, vp, i64, vp, i64, ctypes.POINTER(_Epilogue), vp, sz, vp], i32),
            "qgemm_ptq1_packed_bytes": ([i64, i64], sz),
            "qgemm_ptq1_prepack": ([vp, i64, i64, i64, vp, vp], i32),
            "qgemm_ptq1": ([vp, i64, i64, vp, vp, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_ptq1_prepared": ([vp, i64, i64, vp, vp, vp, i64, vp, i64, vp, sz, vp], i32),
            "qgemm_debug_expand": ([i32, vp, i64, vp, vp], i32),
            "qgemm_get_counters": ([ctypes.POINTER(_Counters)], i32),
            "qgemm_reset_counters": ([], i32),
            "qgemm_get_device_status": ([ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)], i32),
            "qgemm_set_option": ([i32, i64], i32),
            "qgemm_get_option": ([i32], i64),
            "qgemm_set_profile_events": ([vp, vp], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != QGEMM_OK:
        raise QgemmError(rc, lib().qgemm_last_error().decode())


def _ptr(t: torch.Tensor | None, host_ok: bool = False):
    """The address the kernels use.  Device tensors only, except where
    `host_ok`: X, the expert ids and Y may also be pinned host tensors, which
    the kernels read or write across the host link (pageable memory is
    refused here, before anything is launched)."""
    if t is None:
        return None
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError("a CUDA tensor is required here" if not host_ok else
                         "X, ids and Y must be CUDA tensors or pinned host tensors (Tensor.pin_memory())")
    return ctypes.c_void_p(t.data_ptr())


def _device_of(t: torch.Tensor) -> torch.device:
    """Where outputs derived from `t` go: its own device, or the current CUDA
    device for a pinned host tensor."""
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


@dataclasses.dataclass
class Q8K:
    """Q8_K activations as three device planes (row stride K, K/256, K/16)."""
    qs: torch.Tensor      # int8  [M, K]
    d: torch.Tensor       # fp32  [M, K/256]
    bsums: torch.Tensor   # int16 [M, K/16]

    @property
    def M(self) -> int:
        return self.qs.shape[0]

    @property
    def K(self) -> int:
        return self.qs.shape[1]

    @staticmethod
    def empty(M: int, K: int, device="cuda") -> "Q8K":
        return Q8K(torch.empty((M, K), dtype=torch.int8, device=device),
                   torch.empty((M, K // 256), dtype=torch.float32, device=device),
                   torch.empty((M, K // 16), dtype=torch.int16, device=device))


def qgemm_q8k_bytes(M: int, K: int) -> int:
    return int(lib().qgemm_q8k_bytes(M, K))


def q8k_in_buffer(buf: torch.Tensor, M: int, K: int) -> "Q8K":
    """The three Q8_K planes inside one caller-owned buffer of at least
    qgemm_q8k_bytes(M, K) bytes (uint8, 256-B aligned), as views of it."""
    assert buf.dtype == torch.uint8 and buf.is_contiguous()
    assert buf.numel() >= qgemm_q8k_bytes(M, K)
    qs, d, bs = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    _check(lib().qgemm_q8k_planes(_ptr(buf), M, K, ctypes.byref(qs), ctypes.byref(d), ctypes.byref(bs)))
    base = buf.data_ptr()
    o_d, o_bs = d.value - base, bs.value - base
    return Q8K(buf[:M * K].view(torch.int8).view(M, K),
               buf[o_d:o_d + M * (K // 256) * 4].view(torch.float32).view(M, K // 256),
               buf[o_bs:o_bs + M * (K // 16) * 2].view(torch.int16).view(M, K // 16))


def qgemm_q8k_aos_bytes(M: int, K: int) -> int:
    return int(lib().qgemm_q8k_aos_bytes(M, K))


def qgemm_pack_q8k_aos(x: "Q8K", out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Q8K planes -> uint8 [M * K/256 * 292] of 292-byte blocks (d, qs, bsums)."""
    if out is None:
        out = torch.empty(max(qgemm_q8k_aos_bytes(x.M, x.K), 4), dtype=torch.uint8, device=x.qs.device)
    _check(lib().qgemm_pack_q8k_aos(_ptr(x.qs), _ptr(x.d), _ptr(x.bsums), x.M, x.K, _ptr(out), _stream(stream)))
    return out


def qgemm_unpack_q8k_aos(aos: torch.Tensor, M: int, K: int, out: "Q8K | None" = None, stream=None) -> "Q8K":
    """292-byte blocks -> Q8K planes."""
    if out is None:
        out = Q8K.empty(M, K, aos.device)
    _check(lib().qgemm_unpack_q8k_aos(_ptr(aos), M, K, _ptr(out.qs), _ptr(out.d), _ptr(out.bsums), _stream(stream)))
    return out


def qgemm_version() -> int:
    return lib().qgemm_version()


def qgemm_quantize_q8k(x: torch.Tensor, out: Q8K | None = None, stream=None) -> Q8K:
    """fp32 [M, K] (row stride x.stride(0)) -> Q8K planes."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        out = Q8K.empty(M, K, _device_of(x))
    _check(lib().qgemm_quantize_q8k(_ptr(x, True), M, K, x.stride(0), _ptr(out.qs), _ptr(out.d), _ptr(out.bsums),
                                    _stream(stream)))
    return out


def qgemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().qgemm_workspace_bytes(M, N, K))


def _workspace(M, N, K, workspace, device):
    need = qgemm_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace


def qgemm_q4k(w: torch.Tensor, N: int, K: int, x: Q8K, y: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[M, N] = X_q8k @ W_q4k^T.  w: uint8 [N, ldw] device tensor of Q4_K blocks."""
    assert w.dtype == torch.uint8 and w.dim() == 2 and w.stride(1) == 1
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.qs.device)
    workspace = _workspace(M, N, K, workspace, x.qs.device)
    _check(lib().qgemm_q4k(_ptr(w), N, K, w.stride(0), _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True),
                           y.stride(0), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def qgemm_q4k_noalloc(w: torch.Tensor, N: int, K: int, x: Q8K, y: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """qgemm_q4k without a workspace: the library's built-in device scratch is
    used (for callers that cannot allocate; see include/qgemm.h)."""
    assert w.dtype == torch.uint8 and w.dim() == 2 and w.stride(1) == 1
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.qs.device)
    _check(lib().qgemm_q4k_noalloc(_ptr(w), N, K, w.stride(0), _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True),
                                   y.stride(0), _stream(stream)))
    return y


def qgemm_q6k_packed_bytes(N: int, K: int) -> int:
    return int(lib().qgemm_q6k_packed_bytes(N, K))


def qgemm_q6k_prepack(w_aos: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """Q6_K blocks (uint8 [N, ldw]) -> the padded layout qgemm_q6k reads."""
    assert w_aos.dtype == torch.uint8 and w_aos.dim() == 2 and w_aos.stride(1) == 1
    if out is None:
        out = torch.empty(qgemm_q6k_packed_bytes(N, K), dtype=torch.uint8, device=w_aos.device)
    _check(lib().qgemm_q6k_prepack(_ptr(w_aos), N, K, w_aos.stride(0), _ptr(out), _stream(stream)))
    return out


def qgemm_q6k(w_packed: torch.Tensor, N: int, K: int, x: Q8K, y: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.qs.device)
    workspace = _workspace(M, N, K, workspace, x.qs.device)
    _check(lib().qgemm_q6k(_ptr(w_packed), N, K, _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True), y.stride(0),
                           _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def qgemm_quantize_q8k_prep(x: torch.Tensor, workspace: torch.Tensor, out: Q8K | None = None,
                            stream=None) -> Q8K:
    """qgemm_quantize_q8k that also fills `workspace` with the tile GEMM's
    operand planes, for qgemm_q4k_prepared / qgemm_q6k_prepared."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        out = Q8K.empty(M, K, _device_of(x))
    _check(lib().qgemm_quantize_q8k_prep(_ptr(x, True), M, K, x.stride(0), _ptr(out.qs), _ptr(out.d), _ptr(out.bsums),
                                         _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def qgemm_q4k_f32(w: torch.Tensor, N: int, K: int, x: torch.Tensor, out: Q8K | None = None,
                  y: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[M, N] = Q8_K(x) @ W_q4k^T from fp32 x [M, K]; the Q8_K planes of x go
    to `out` (allocated if None).  The workspace is needed only above the
    small-M path (allocated if None)."""
    assert w.dtype == torch.uint8 and w.dim() == 2 and w.stride(1) == 1
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    dev = _device_of(x)
    if out is None:
        out = Q8K.empty(M, K, dev)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    workspace = _workspace(M, N, K, workspace, dev)
    _check(lib().qgemm_q4k_f32(_ptr(w), N, K, w.stride(0), _ptr(x, True), x.stride(0), M, _ptr(out.qs), _ptr(out.d),
                               _ptr(out.bsums), _ptr(y, True), y.stride(0), _ptr(workspace), workspace.numel(),
                               _stream(stream)))
    return y


def qgemm_q6k_f32(w_packed: torch.Tensor, N: int, K: int, x: torch.Tensor, out: Q8K | None = None,
                  y: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qgemm_q4k_f32 for repacked Q6_K weights."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    dev = _device_of(x)
    if out is None:
        out = Q8K.empty(M, K, dev)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    workspace = _workspace(M, N, K, workspace, dev)
    _check(lib().qgemm_q6k_f32(_ptr(w_packed), N, K, _ptr(x, True), x.stride(0), M, _ptr(out.qs), _ptr(out.d),
                               _ptr(out.bsums), _ptr(y, True), y.stride(0), _ptr(workspace), workspace.numel(),
                               _stream(stream)))
    return y


def qgemm_ptq1_f32(w_packed: torch.Tensor, N: int, K: int, x: torch.Tensor, out: Q8K | None = None,
                   y: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qgemm_q4k_f32 for repacked PTQ1_0 weights (always the tile GEMM)."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    dev = _device_of(x)
    if out is None:
        out = Q8K.empty(M, K, dev)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    workspace = _workspace(M, N, K, workspace, dev)
    _check(lib().qgemm_ptq1_f32(_ptr(w_packed), N, K, _ptr(x, True), x.stride(0), M, _ptr(out.qs), _ptr(out.d),
                                _ptr(out.bsums), _ptr(y, True), y.stride(0), _ptr(workspace), workspace.numel(),
                                _stream(stream)))
    return y


def qgemm_q4k_prepared(w: torch.Tensor, N: int, K: int, x: Q8K, workspace: torch.Tensor,
                       y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qgemm_q4k with a workspace filled by qgemm_quantize_q8k_prep from `x`."""
    assert w.dtype == torch.uint8 and w.dim() == 2 and w.stride(1) == 1
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.qs.device)
    _check(lib().qgemm_q4k_prepared(_ptr(w), N, K, w.stride(0), _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True),
                                    y.stride(0), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def qgemm_q6k_prepared(w_packed: torch.Tensor, N: int, K: int, x: Q8K, workspace: torch.Tensor,
                       y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qgemm_q6k with a workspace filled by qgemm_quantize_q8k_prep from `x`."""
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.qs.device)
    _check(lib().qgemm_q6k_prepared(_ptr(w_packed), N, K, _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True),
                                    y.stride(0), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def qgemm_id_workspace_bytes(M: int, top_k: int, experts: int, K: int) -> int:
    return int(lib().qgemm_id_workspace_bytes(M, top_k, experts, K))


def qgemm_q4k_id(w: torch.Tensor, experts: int, N: int, K: int, x: Q8K, ids: torch.Tensor,
                 y: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Expert-routed GEMM: w uint8 [experts * N, ldw] Q4_K rows (expert e = rows e*N ..),
    ids int32 [M, top_k]; returns Y fp32 [M * top_k, N], row i*top_k + s = W_{ids[i, s]} x_i."""
    assert w.dtype == torch.uint8 and w.dim() == 2 and w.stride(1) == 1
    assert ids.dtype == torch.int32 and ids.dim() == 2 and ids.is_contiguous()
    M, top_k = ids.shape
    assert M == x.M
    if y is None:
        y = torch.empty((M * top_k, N), dtype=torch.float32, device=x.qs.device)
    if workspace is None:
        workspace = torch.empty(max(qgemm_id_workspace_bytes(M, top_k, experts, K), 256), dtype=torch.uint8,
                                device=x.qs.device)
    _check(lib().qgemm_q4k_id(_ptr(w), experts, N, K, w.stride(0), _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M,
                              _ptr(ids, True), top_k, _ptr(y, True), y.stride(0), _ptr(workspace), workspace.numel(),
                              _stream(stream)))
    return y


def qgemm_q6k_id(w_packed: torch.Tensor, experts: int, N: int, K: int, x: Q8K, ids: torch.Tensor,
                 y: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """As qgemm_q4k_id, with the experts' Q6_K rows repacked by qgemm_q6k_prepack (N = experts * N)."""
    assert ids.dtype == torch.int32 and ids.dim() == 2 and ids.is_contiguous()
    M, top_k = ids.shape
    assert M == x.M
    if y is None:
        y = torch.empty((M * top_k, N), dtype=torch.float32, device=x.qs.device)
    if workspace is None:
        workspace = torch.empty(max(qgemm_id_workspace_bytes(M, top_k, experts, K), 256), dtype=torch.uint8,
                                device=x.qs.device)
    _check(lib().qgemm_q6k_id(_ptr(w_packed), experts, N, K, _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(ids, True),
                              top_k, _ptr(y, True), y.stride(0), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


_OUT_TYPES = {torch.float32: QGEMM_OUT_F32, torch.float16: QGEMM_OUT_F16, torch.bfloat16: QGEMM_OUT_BF16}


def _epilogue(out_dtype, bias, activation) -> _Epilogue:
    if bias is not None:
        assert bias.dtype == torch.float32 and bias.is_contiguous()
    return _Epilogue(_OUT_TYPES[out_dtype], int(activation), None if bias is None else bias.data_ptr())


def qgemm_q4k_ex(w: torch.Tensor, N: int, K: int, x: Q8K, out_dtype=torch.float32, bias: torch.Tensor | None = None,
                 activation: int = QGEMM_ACT_NONE, y: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out_dtype(act(X_q8k @ W_q4k^T + bias)); out_dtype float32 / float16 / bfloat16."""
    assert w.dtype == torch.uint8 and w.dim() == 2 and w.stride(1) == 1
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.qs.device)
    assert y.dtype == out_dtype
    workspace = _workspace(M, N, K, workspace, x.qs.device)
    ep = _epilogue(out_dtype, bias, activation)
    _check(lib().qgemm_q4k_ex(_ptr(w), N, K, w.stride(0), _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True),
                              y.stride(0), ctypes.byref(ep), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def qgemm_q6k_ex(w_packed: torch.Tensor, N: int, K: int, x: Q8K, out_dtype=torch.float32,
                 bias: torch.Tensor | None = None, activation: int = QGEMM_ACT_NONE, y: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """As qgemm_q4k_ex with repacked Q6_K weights."""
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.qs.device)
    assert y.dtype == out_dtype
    workspace = _workspace(M, N, K, workspace, x.qs.device)
    ep = _epilogue(out_dtype, bias, activation)
    _check(lib().qgemm_q6k_ex(_ptr(w_packed), N, K, _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True), y.stride(0),
                              ctypes.byref(ep), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


PTQ1_BLOCK_BYTES = 28


def qgemm_ptq1_prepack(w: torch.Tensor, N: int, K: int, stream=None) -> torch.Tensor:
    """PTQ1_0 rows uint8 [N, ldw] (28-byte blocks) -> repacked uint8 [N, K/4] (32-byte blocks)."""
    assert w.dtype == torch.uint8 and w.dim() == 2 and w.stride(1) == 1
    out = torch.empty((N, K // 4), dtype=torch.uint8, device=w.device)
    _check(lib().qgemm_ptq1_prepack(_ptr(w), N, K, w.stride(0), _ptr(out), _stream(stream)))
    return out


def qgemm_ptq1(w_packed: torch.Tensor, N: int, K: int, x: Q8K, y: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[M, N] = X_q8k @ W_ptq1^T from qgemm_ptq1_prepack's output."""
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.qs.device)
    workspace = _workspace(M, N, K, workspace, x.qs.device)
    _check(lib().qgemm_ptq1(_ptr(w_packed), N, K, _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True), y.stride(0),
                            _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def qgemm_ptq1_prepared(w_packed: torch.Tensor, N: int, K: int, x: Q8K, workspace: torch.Tensor,
                        y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qgemm_ptq1 from a workspace that qgemm_quantize_q8k_prep filled for the same X."""
    M = x.M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.qs.device)
    _check(lib().qgemm_ptq1_prepared(_ptr(w_packed), N, K, _ptr(x.qs), _ptr(x.d), _ptr(x.bsums), M, _ptr(y, True),
                                     y.stride(0), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y


def qgemm_debug_expand(wtype: int, blocks: torch.Tensor, nblocks: int, stream=None) -> torch.Tensor:
    """The tile GEMM's weight expansion of `nblocks` superblock rows (test
    diagnostic): uint32 [nblocks, QGEMM_DEBUG_EXPAND_BYTES / 4] records."""
    out = torch.empty((max(nblocks, 1), QGEMM_DEBUG_EXPAND_BYTES // 4), dtype=torch.int32, device=blocks.device)
    _check(lib().qgemm_debug_expand(wtype, _ptr(blocks), nblocks, _ptr(out), _stream(stream)))
    return out[:nblocks]


def qgemm_get_counters() -> dict:
    c = _Counters()
    _check(lib().qgemm_get_counters(ctypes.byref(c)))
    return {n: int(getattr(c, n)) for n, _ in _Counters._fields_}


def qgemm_reset_counters() -> None:
    _check(lib().qgemm_reset_counters())


def qgemm_get_device_status() -> tuple[int, int]:
    """(bits, site) of the current device's status word, which is then
    cleared.  A set bit is reported, not raised (the C call returns
    QGEMM_ETIMEOUT / QGEMM_EDEVICE for it); other failures raise."""
    bits, site = ctypes.c_uint32(0), ctypes.c_uint32(0)
    rc = lib().qgemm_get_device_status(ctypes.byref(bits), ctypes.byref(site))
    if rc not in (QGEMM_OK, QGEMM_ETIMEOUT, QGEMM_EDEVICE):
        _check(rc)
    return int(bits.value), int(site.value)


def qgemm_device_status_code() -> tuple[int, int, int]:
    """(return code, bits, site) of qgemm_get_device_status, unraised."""
    bits, site = ctypes.c_uint32(0), ctypes.c_uint32(0)
    rc = lib().qgemm_get_device_status(ctypes.byref(bits), ctypes.byref(site))
    return int(rc), int(bits.value), int(site.value)


def qgemm_set_option(option: int, value: int) -> None:
    _check(lib().qgemm_set_option(option, value))


def qgemm_get_option(option: int) -> int:
    return int(lib().qgemm_get_option(option))


def qgemm_set_profile_events(before=None, after=None) -> None:
    """torch.cuda.Event objects (already created, e.g. recorded once) or None."""
    def h(ev):
        return None if ev is None else ctypes.c_void_p(ev.cuda_event)
    _check(lib().qgemm_set_profile_events(h(before), h(after)))

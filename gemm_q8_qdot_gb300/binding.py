"""Thin ctypes binding of libpq (include/pq.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module turns
torch CUDA tensors into device pointers, sizes and the current stream, calls
the C entry point of the same name and raises PQError on a non-zero status.
There is no CPU fallback: if libpq.so cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

PQ_OK = 0
PQ_ERR_INVALID_ARG = -1
PQ_ERR_SHAPE = -2
PQ_ERR_ALIGN = -3
PQ_ERR_CUDA = -4
PQ_ERR_TIMEOUT = -5
PQ_ERR_UNSUPPORTED = -6
PQ_ERR_SCRATCH = -7

PATH_AUTO, PATH_SIMT, PATH_TC, PATH_MMA = 0, 1, 2, 3
WS_N_KB, WS_KB_N = 0, 1

EXPORTS = ("pq_quantize_q8_0", "pq_qdot_q8_0", "pq_qdot_q8_0_ex", "pq_quantize_qdot_q8_0",
           "pq_last_cuda_error",
           "pq_quantize_qdot_q8_0_noalloc", "pq_quantize_qdot_q8_0_host", "pq_qdot_q8_0_blocksums", "pq_q50_qdot",
           "pq_quantize_q50_qdot", "pq_q50_blocksums", "pq_check_device", "pq_strerror", "pq_version")

_lib: ctypes.CDLL | None = None


class PQError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libpq.so (built by __graft_entry__.build() / gemm_q8_qdot_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libpq.so not built ({path}); run gemm_q8_qdot_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.pq_quantize_q8_0.argtypes = [vp, vp, vp, i64, i64, vp]
    lib.pq_qdot_q8_0.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.pq_qdot_q8_0_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, vp]
    lib.pq_quantize_qdot_q8_0.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_last_cuda_error.argtypes = []
    lib.pq_debug_stream_read.argtypes = [vp, vp, i64, i64, vp, i32, vp]
    lib.pq_quantize_qdot_q8_0_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_quantize_qdot_q8_0_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_qdot_q8_0_blocksums.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_q50_qdot.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_quantize_q50_qdot.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_q50_blocksums.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    lib.pq_check_device.argtypes = [vp]
    lib.pq_strerror.argtypes = [i32]
    lib.pq_strerror.restype = ctypes.c_char_p
    lib.pq_version.argtypes = []
    for fn in ("pq_quantize_q8_0", "pq_qdot_q8_0", "pq_qdot_q8_0_ex", "pq_quantize_qdot_q8_0",
               "pq_last_cuda_error", "pq_debug_stream_read",
               "pq_quantize_qdot_q8_0_noalloc", "pq_quantize_qdot_q8_0_host", "pq_qdot_q8_0_blocksums",
               "pq_q50_qdot", "pq_quantize_q50_qdot", "pq_q50_blocksums", "pq_check_device", "pq_version"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().pq_strerror(int(code)).decode()
    except RuntimeError:
        return f"pq_status {code}"


# The current stream's raw handle without building a torch.cuda.Stream object
# (about 3 us per call otherwise, as much as the library call itself).
_raw_stream_of = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    """The stream argument as a raw handle; None = the current device's current stream
    (the device the library launches on)."""
    if stream is None:
        if _raw_stream_of is not None:
            return _raw_stream_of(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("expected a contiguous (row-major) CUDA tensor")
    return t.data_ptr()


def _check(code: int, where: str) -> None:
    if code != PQ_OK:
        raise PQError(code, where)


def quantize_q8_0(x: torch.Tensor, q: torch.Tensor | None = None, s: torch.Tensor | None = None,
                  stream=None):
    """f32 [rows, K] -> (q int8 [rows, K], s f32 [rows, K/32]) via pq_quantize_q8_0."""
    if x.dtype != torch.float32:
        raise TypeError("x must be float32")
    x2 = x if x.dim() == 2 else x.reshape(-1, x.shape[-1])
    rows, K = x2.shape
    if q is None:
        q = torch.empty((rows, K), dtype=torch.int8, device=x.device)
    if s is None:
        s = torch.empty((rows, K // 32 if K % 32 == 0 else 0), dtype=torch.float32, device=x.device)
    _check(load().pq_quantize_q8_0(_ptr(x2), _ptr(q), _ptr(s), rows, K, _stream(stream)), "pq_quantize_q8_0")
    return q, s


def qdot_q8_0(A, AS, W, WS, C=None, stream=None):
    """C[M, N] = qdot_t(A, AS, W, WS) via pq_qdot_q8_0 (kernel chosen by M)."""
    M, K = A.shape
    N = W.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(load().pq_qdot_q8_0(_ptr(A), _ptr(AS), _ptr(W), _ptr(WS), _ptr(C), M, N, K, _stream(stream)),
           "pq_qdot_q8_0")
    return C


def qdot_q8_0_ex(A, AS, W, WS, C=None, ws_layout: int = WS_N_KB, path: int = PATH_AUTO, stream=None):
    """pq_qdot_q8_0_ex: explicit weight-scale layout and kernel path."""
    M, K = A.shape
    N = W.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(load().pq_qdot_q8_0_ex(_ptr(A), _ptr(AS), _ptr(W), _ptr(WS), _ptr(C), M, N, K,
                                  int(ws_layout), int(path), _stream(stream)), "pq_qdot_q8_0_ex")
    return C


def quantize_qdot_q8_0(x, W, WS, C=None, A=None, AS=None, ws_layout: int = WS_N_KB, stream=None):
    """One decode step via pq_quantize_qdot_q8_0: C = qdot_t(quantize(x), W); A/AS optionally
    receive the quantized rows (both or neither; without them the library keeps the rows in
    its own workspace)."""
    if x.dtype != torch.float32:
        raise TypeError("x must be float32")
    M, K = x.shape
    N = W.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(load().pq_quantize_qdot_q8_0(_ptr(x), _ptr(A), _ptr(AS), _ptr(W), _ptr(WS), _ptr(C), M, N, K,
                                        int(ws_layout), _stream(stream)), "pq_quantize_qdot_q8_0")
    return C


def debug_stream_read(W, WS, out=None, early: bool = False, stream=None):
    """Test-only: the decode step's weight stream without its arithmetic (pq_debug_stream_read);
    out[row] receives a checksum of the row."""
    rows, K = W.shape
    if out is None:
        out = torch.empty((rows,), dtype=torch.float32, device=W.device)
    _check(load().pq_debug_stream_read(_ptr(W), _ptr(WS), rows, K, _ptr(out), int(early), _stream(stream)),
           "pq_debug_stream_read")
    return out


def quantize_qdot_q8_0_host(x_host, W, WS, C_host, ws_layout: int = WS_N_KB, stream=None):
    """pq_quantize_qdot_q8_0_host: one decode step from host x_host [M, K] f32 into host C_host
    [M, N] f32 (a page-locked C_host is written in place by the kernels, a pageable one through
    a copy); enqueued on the stream, which the caller synchronizes before reading C_host."""
    if x_host.dtype != torch.float32 or C_host.dtype != torch.float32:
        raise TypeError("x_host and C_host must be float32")
    if x_host.is_cuda or C_host.is_cuda:
        raise ValueError("x_host and C_host must be host tensors")
    if not (x_host.is_contiguous() and C_host.is_contiguous()):
        raise ValueError("x_host and C_host must be contiguous")
    M, K = x_host.shape
    N = W.shape[0]
    if tuple(C_host.shape) != (M, N):
        raise ValueError("C_host must be [M, N]")
    _check(load().pq_quantize_qdot_q8_0_host(x_host.data_ptr(), _ptr(W), _ptr(WS), C_host.data_ptr(), M, N, K,
                                             int(ws_layout), _stream(stream)), "pq_quantize_qdot_q8_0_host")
    return C_host


def quantize_qdot_q8_0_noalloc(x, W, WS, C=None, ws_layout: int = WS_N_KB, stream=None):
    """pq_quantize_qdot_q8_0_noalloc: the one-call step with the quantized rows in the library's
    fixed device array instead of an allocated workspace (for callers that cannot allocate)."""
    if x.dtype != torch.float32:
        raise TypeError("x must be float32")
    M, K = x.shape
    N = W.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(load().pq_quantize_qdot_q8_0_noalloc(_ptr(x), _ptr(W), _ptr(WS), _ptr(C), M, N, K, int(ws_layout),
                                                _stream(stream)), "pq_quantize_qdot_q8_0_noalloc")
    return C


def qdot_q8_0_blocksums(A, W, S=None, path: int = PATH_SIMT, stream=None):
    """int32 block sums S[M, N, K/32] by the engine of `path` (verification entry point)."""
    M, K = A.shape
    N = W.shape[0]
    if S is None:
        S = torch.empty((M, N, K // 32), dtype=torch.int32, device=A.device)
    _check(load().pq_qdot_q8_0_blocksums(_ptr(A), _ptr(W), _ptr(S), M, N, K, int(path), _stream(stream)),
           "pq_qdot_q8_0_blocksums")
    return S


def q50_qdot(A, AS, W5, WS, C=None, ws_layout: int = WS_N_KB, stream=None):
    """pq_q50_qdot: C = q50_qdot_t(A, AS, W5, WS); W5 uint8 [N, K/32 * 20] Q5_0 blocks."""
    M, K = A.shape
    N = W5.shape[0]
    if W5.dtype != torch.uint8 or W5.shape[1] != K // 32 * 20:
        raise ValueError("W5 must be uint8 [N, K/32 * 20]")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(load().pq_q50_qdot(_ptr(A), _ptr(AS), _ptr(W5), _ptr(WS), _ptr(C), M, N, K, int(ws_layout),
                              _stream(stream)), "pq_q50_qdot")
    return C


def quantize_q50_qdot(x, W5, WS, C=None, A=None, AS=None, ws_layout: int = WS_N_KB, stream=None):
    """One decode step against Q5_0 weights via pq_quantize_q50_qdot: C = q50_qdot_t(quantize(x), W5);
    A/AS optionally receive the quantized rows (both or neither)."""
    if x.dtype != torch.float32:
        raise TypeError("x must be float32")
    M, K = x.shape
    N = W5.shape[0]
    if W5.dtype != torch.uint8 or W5.shape[1] != K // 32 * 20:
        raise ValueError("W5 must be uint8 [N, K/32 * 20]")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(load().pq_quantize_q50_qdot(_ptr(x), _ptr(A), _ptr(AS), _ptr(W5), _ptr(WS), _ptr(C), M, N, K,
                                       int(ws_layout), _stream(stream)), "pq_quantize_q50_qdot")
    return C


def q50_blocksums(A, W5, S=None, stream=None):
    """int32 block sums of pq_q50_qdot (verification entry point)."""
    M, K = A.shape
    N = W5.shape[0]
    if S is None:
        S = torch.empty((M, N, K // 32), dtype=torch.int32, device=A.device)
    _check(load().pq_q50_blocksums(_ptr(A), _ptr(W5), _ptr(S), M, N, K, _stream(stream)), "pq_q50_blocksums")
    return S


def check_device(stream=None) -> None:
    """Synchronizes the stream and raises PQError if a bounded on-device wait gave up."""
    _check(load().pq_check_device(_stream(stream)), "pq_check_device")

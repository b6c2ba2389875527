"""block_quantized_matmul_gb300 -- Python binding of libqmm (include/qmm.h).

Matrix multiply over block-32 quantized weights (Q4_0, Q8_0, IQ4_NL; also MXFP4, Q4_1 and the
Q4_K super-blocks) stored in the 32-row tiled layout of "Hexagon backend developer details" ("Tiled
Weight Formats") or in flat GGML rows, with activations dynamically quantized to Q8_0 blocks, on
one GB300 (sm_103a).

This module only marshals arguments: every function takes torch CUDA tensors (PyTorch provides the
device memory and the stream; the fused decode call also takes pinned host tensors for x and y),
passes raw addresses and sizes through ctypes, and raises QmmError on any status other than QMM_OK.
All computation runs in the CUDA kernels of libqmm.so; there is no CPU fallback, and the first call
fails loudly if the library is missing.

A decode step over a weight w (fp32 [N, K] on the GPU):

    flat = torch.empty(flat_size("q4_0", K, N), dtype=torch.uint8, device="cuda")
    tiled = torch.empty(tiled_size("q4_0", K, N), dtype=torch.uint8, device="cuda")
    qmm_quantize_weight("q4_0", w, N, K, K, flat)        # load time
    qmm_repack("q4_0", flat, K, N, tiled)               # load time
    qmm_matmul_f32("q4_0", tiled, K, N, x, K, M, y, N)   # y[M, N] = Q8_0(x[M, K]) @ W^T

Prefill shapes: qmm_quantize_act, then qmm_matmul_ws with a workspace of matmul_workspace_size(M, K)
bytes (or qmm_matmul, which needs none).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "Q4_0", "Q8_0", "IQ4_NL", "MXFP4", "Q4_1", "Q4_K", "TYPES", "QmmError", "lib", "library_path",
    "block_size", "tile_size", "tiled_size", "flat_size", "iq4nl_table", "decode_max_m",
    "qmm_quantize_weight", "qmm_repack", "qmm_unpack", "qmm_quantize_act", "qmm_matmul",
    "qmm_matmul_path", "qmm_matmul_f32", "qmm_matmul_flat", "qmm_device_status", "PATH_AUTO", "PATH_MATVEC", "PATH_GEMM",
    "matmul_workspace_size", "qmm_matmul_ws", "qmm_matmul_noalloc", "matmul_noalloc_max_workspace",
    "qmm_selftest_timeout",
]

Q4_0, Q8_0, IQ4_NL, MXFP4, Q4_1, Q4_K = 0, 1, 2, 3, 4, 5
TYPES = {"q4_0": Q4_0, "q8_0": Q8_0, "iq4_nl": IQ4_NL, "mxfp4": MXFP4, "q4_1": Q4_1, "q4_k": Q4_K}
PATH_AUTO, PATH_MATVEC, PATH_GEMM = 0, 1, 2
_STATUS = {0: "QMM_OK", 1: "QMM_ERR_INVALID_ARG", 2: "QMM_ERR_UNSUPPORTED", 3: "QMM_ERR_MISALIGNED",
           4: "QMM_ERR_CUDA", 5: "QMM_ERR_TIMEOUT", 6: "QMM_ERR_RANGE", 7: "QMM_ERR_BOUNDS"}

_HERE = os.path.dirname(os.path.abspath(__file__))
# QMM_DEBUG=1 in the environment selects the build with device bounds checks (libqmm_debug.so)
library_path = os.path.join(_HERE, "libqmm_debug.so" if os.environ.get("QMM_DEBUG") == "1" else "libqmm.so")
_lib = None


class QmmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)}")


def lib():
    """Load libqmm.so (built by build.py / __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise ImportError(f"libqmm.so not built at {library_path}; run `python -m block_quantized_matmul_gb300.build`")
        L = ctypes.CDLL(library_path)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        L.qmm_status_str.argtypes = [i32]
        L.qmm_status_str.restype = ctypes.c_char_p
        for fn in ("qmm_block_size", "qmm_tile_size"):
            getattr(L, fn).argtypes = [i32]
            getattr(L, fn).restype = sz
        for fn in ("qmm_tiled_size", "qmm_flat_size"):
            getattr(L, fn).argtypes = [i32, i64, i64]
            getattr(L, fn).restype = sz
        L.qmm_iq4nl_table.argtypes = [vp]
        L.qmm_iq4nl_table.restype = None
        L.qmm_decode_max_m.argtypes = []
        L.qmm_decode_max_m.restype = i64
        L.qmm_quantize_weight.argtypes = [i32, vp, i64, i64, i64, vp, vp]
        L.qmm_repack.argtypes = [i32, vp, i64, i64, vp, vp]
        L.qmm_unpack.argtypes = [i32, vp, i64, i64, vp, vp]
        L.qmm_quantize_act.argtypes = [vp, i64, i64, i64, vp, vp, vp]
        L.qmm_matmul.argtypes = [i32, vp, i64, i64, vp, vp, i64, vp, i64, vp]
        L.qmm_matmul_f32.argtypes = [i32, vp, i64, i64, vp, i64, i64, vp, i64, vp]
        L.qmm_matmul_path.argtypes = [i32, vp, i64, i64, vp, vp, i64, vp, i64, i32, vp]
        L.qmm_matmul_flat.argtypes = [i32, vp, i64, i64, vp, vp, i64, vp, i64, vp]
        L.qmm_device_status.argtypes = [vp]
        L.qmm_selftest_timeout.argtypes = [i32, ctypes.c_uint64, vp, vp]
        L.qmm_matmul_workspace_size.argtypes = [i64, i64]
        L.qmm_matmul_workspace_size.restype = sz
        L.qmm_matmul_ws.argtypes = [i32, vp, i64, i64, vp, vp, i64, vp, i64, vp, sz, vp]
        L.qmm_matmul_noalloc.argtypes = [i32, vp, i64, i64, vp, vp, i64, vp, i64, vp]
        L.qmm_matmul_noalloc_max_workspace.argtypes = []
        L.qmm_matmul_noalloc_max_workspace.restype = sz
        L.qmm_matmul_f32_workspace_size.argtypes = [i64, i64]
        L.qmm_matmul_f32_workspace_size.restype = sz
        L.qmm_matmul_f32_ws.argtypes = [i32, vp, i64, i64, vp, i64, i64, vp, i64, vp, sz, vp]
        for fn in ("qmm_quantize_weight", "qmm_repack", "qmm_unpack", "qmm_quantize_act", "qmm_matmul",
                   "qmm_matmul_path", "qmm_device_status", "qmm_matmul_ws", "qmm_matmul_noalloc", "qmm_matmul_f32",
                   "qmm_matmul_flat", "qmm_selftest_timeout", "qmm_matmul_f32_ws"):
            getattr(L, fn).restype = i32
        _lib = L
    return _lib


def _t(type_) -> int:
    return TYPES[type_] if isinstance(type_, str) else int(type_)


def _ptr(x) -> int | None:
    """Address of a CUDA tensor or of a page-locked (pinned) host tensor, which the GPU reads and
    writes directly (or a raw integer address)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda and not x.is_pinned():
        raise ValueError("libqmm takes CUDA tensors or pinned host tensors only")
    return x.data_ptr()


def _ptr_located(x) -> int | None:
    """Address of a tensor for the calls that check on their own where x and y point (device or
    page-locked host memory; pageable memory is refused by the library): no host-side query here."""
    if x is None or isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise QmmError(fn, st)


def block_size(type_) -> int:
    return int(lib().qmm_block_size(_t(type_)))


def tile_size(type_) -> int:
    return int(lib().qmm_tile_size(_t(type_)))


def tiled_size(type_, K: int, N: int) -> int:
    return int(lib().qmm_tiled_size(_t(type_), K, N))


def flat_size(type_, K: int, N: int) -> int:
    return int(lib().qmm_flat_size(_t(type_), K, N))


def iq4nl_table() -> list[int]:
    buf = (ctypes.c_int8 * 16)()
    lib().qmm_iq4nl_table(ctypes.cast(buf, ctypes.c_void_p))
    return list(buf)


def decode_max_m() -> int:
    return int(lib().qmm_decode_max_m())


def qmm_quantize_weight(type_, w, N: int, K: int, ldw: int, w_flat, stream=None) -> None:
    _check("qmm_quantize_weight",
           lib().qmm_quantize_weight(_t(type_), _ptr(w), N, K, ldw, _ptr(w_flat), _stream(stream)))


def qmm_repack(type_, w_flat, K: int, N: int, w_tiled, stream=None) -> None:
    _check("qmm_repack", lib().qmm_repack(_t(type_), _ptr(w_flat), K, N, _ptr(w_tiled), _stream(stream)))


def qmm_unpack(type_, w_tiled, K: int, N: int, w_flat, stream=None) -> None:
    _check("qmm_unpack", lib().qmm_unpack(_t(type_), _ptr(w_tiled), K, N, _ptr(w_flat), _stream(stream)))


def qmm_quantize_act(x, M: int, K: int, ldx: int, a_q, a_d, stream=None) -> None:
    _check("qmm_quantize_act",
           lib().qmm_quantize_act(_ptr(x), M, K, ldx, _ptr(a_q), _ptr(a_d), _stream(stream)))


def qmm_matmul(type_, w_tiled, K: int, N: int, a_q, a_d, M: int, y, ldy: int, stream=None) -> None:
    _check("qmm_matmul", lib().qmm_matmul(_t(type_), _ptr(w_tiled), K, N, _ptr(a_q), _ptr(a_d), M, _ptr(y), ldy,
                                          _stream(stream)))


def qmm_matmul_f32(type_, w_tiled, K: int, N: int, x, ldx: int, M: int, y, ldy: int, stream=None) -> None:
    _check("qmm_matmul_f32", lib().qmm_matmul_f32(_t(type_), _ptr(w_tiled), K, N, _ptr_located(x), ldx, M,
                                                  _ptr_located(y), ldy, _stream(stream)))


def matmul_f32_workspace_size(M: int, K: int) -> int:
    return int(lib().qmm_matmul_f32_workspace_size(M, K))


def qmm_matmul_f32_ws(type_, w_tiled, K: int, N: int, x, ldx: int, M: int, y, ldy: int, workspace,
                      workspace_bytes: int, stream=None) -> None:
    _check("qmm_matmul_f32_ws", lib().qmm_matmul_f32_ws(_t(type_), _ptr(w_tiled), K, N, _ptr_located(x), ldx, M,
                                                        _ptr_located(y), ldy, _ptr(workspace), int(workspace_bytes),
                                                        _stream(stream)))


def qmm_matmul_flat(type_, w_flat, K: int, N: int, a_q, a_d, M: int, y, ldy: int, stream=None) -> None:
    _check("qmm_matmul_flat", lib().qmm_matmul_flat(_t(type_), _ptr(w_flat), K, N, _ptr(a_q), _ptr(a_d), M, _ptr(y),
                                                    ldy, _stream(stream)))


def qmm_matmul_path(type_, w_tiled, K: int, N: int, a_q, a_d, M: int, y, ldy: int, path: int,
                    stream=None) -> None:
    _check("qmm_matmul_path", lib().qmm_matmul_path(_t(type_), _ptr(w_tiled), K, N, _ptr(a_q), _ptr(a_d), M,
                                                    _ptr(y), ldy, int(path), _stream(stream)))


def matmul_workspace_size(M: int, K: int) -> int:
    return int(lib().qmm_matmul_workspace_size(M, K))


def qmm_matmul_ws(type_, w_tiled, K: int, N: int, a_q, a_d, M: int, y, ldy: int, workspace, workspace_bytes: int,
                  stream=None) -> None:
    _check("qmm_matmul_ws", lib().qmm_matmul_ws(_t(type_), _ptr(w_tiled), K, N, _ptr(a_q), _ptr(a_d), M, _ptr(y), ldy,
                                                _ptr(workspace), int(workspace_bytes), _stream(stream)))


def qmm_matmul_noalloc(type_, w_tiled, K: int, N: int, a_q, a_d, M: int, y, ldy: int, stream=None) -> None:
    """For callers that cannot allocate device memory: the tensor-core path's workspace is the
    library's fixed per-device scratch array (see include/qmm.h); overlapping calls race on it."""
    _check("qmm_matmul_noalloc", lib().qmm_matmul_noalloc(_t(type_), _ptr(w_tiled), K, N, _ptr(a_q), _ptr(a_d), M,
                                                          _ptr(y), ldy, _stream(stream)))


def matmul_noalloc_max_workspace() -> int:
    return int(lib().qmm_matmul_noalloc_max_workspace())


def qmm_device_status(stream=None) -> int:
    """Synchronize the stream, then return and clear the device status (0 = ok, 5 = timeout)."""
    return int(lib().qmm_device_status(_stream(stream)))


def qmm_selftest_timeout(unit: int, limit_ns: int, flags, stream=None) -> None:
    """Test hook: one CTA whose bounded waits run out on purpose (unit 0: decode kernels' helper,
    1: the GEMM's); afterwards qmm_device_status() reports the timeout (see include/qmm.h)."""
    _check("qmm_selftest_timeout", lib().qmm_selftest_timeout(int(unit), int(limit_ns), _ptr(flags), _stream(stream)))

"""CPU oracle for block-32 quantized matmul over tiled weights -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The product library (``block_quantized_matmul_gb300``) never imports, links or calls
it, and it shares no code with the product: the arithmetic lives in ``oracle/oracle.c`` (plain C,
``-O2 -fno-fast-math -ffp-contract=off``), compiled into ``oracle/liboracle.so`` by
``oracle.build()``; this module only marshals numpy arrays through ctypes.

What it follows ("Hexagon backend developer details", "Tiled Weight Formats"): the tile grid of
"Tile Dimensions and Grid Layout", the Q4_0 / Q8_0 / IQ4_NL / MXFP4 / Q4_1 tile byte layouts of
"Block-32 Quantized Formats" and the Q4_K tile of "K-Quants Formats".  The readings taken where the pages are silent are listed in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_0, Q8_0, IQ4_NL, MXFP4, Q4_1, Q4_K = 0, 1, 2, 3, 4, 5
TYPES = {"q4_0": Q4_0, "q8_0": Q8_0, "iq4_nl": IQ4_NL, "mxfp4": MXFP4, "q4_1": Q4_1, "q4_k": Q4_K}

_HERE = os.path.dirname(os.path.abspath(__file__))
# QMM_ORACLE_SRC points the module at another copy of the C source (the pin-strength test builds
# copies with one planted mistake each); the library is then built next to that copy.
_SRC = os.environ.get("QMM_ORACLE_SRC") or os.path.join(_HERE, "oracle.c")
_LIB = os.path.splitext(_SRC)[0] + ".so" if os.environ.get("QMM_ORACLE_SRC") else os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc); returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f32.restype = ctypes.c_float
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_e8m0_to_f16_bits.argtypes = [i32]
            lib.orc_e8m0_to_f16_bits.restype = ctypes.c_uint16
            for fn in ("orc_block_bytes", "orc_tile_bytes"):
                getattr(lib, fn).argtypes = [i32]
                getattr(lib, fn).restype = i64
            lib.orc_row_bytes.argtypes = [i32, i64]
            lib.orc_row_bytes.restype = i64
            lib.orc_tile_index.argtypes = [i64, i64, i64]
            lib.orc_tile_index.restype = i64
            lib.orc_tiled_bytes.argtypes = [i32, i64, i64]
            lib.orc_tiled_bytes.restype = i64
            lib.orc_quantize_block_q8_0.argtypes = [vp, vp, vp]
            lib.orc_quantize_block_q8_0.restype = None
            lib.orc_quantize_rows.argtypes = [i32, vp, i64, i64, vp, vp]
            lib.orc_quantize_rows.restype = None
            lib.orc_dequantize_flat.argtypes = [i32, vp, i64, i64, vp, vp]
            lib.orc_dequantize_flat.restype = None
            lib.orc_repack.argtypes = [i32, vp, i64, i64, vp]
            lib.orc_repack.restype = None
            lib.orc_unpack.argtypes = [i32, vp, i64, i64, vp]
            lib.orc_unpack.restype = None
            lib.orc_quantize_act.argtypes = [vp, i64, i64, i64, vp, vp]
            lib.orc_quantize_act.restype = None
            lib.orc_matmul.argtypes = [i32, vp, i64, i64, vp, vp, i64, vp, vp, vp]
            lib.orc_matmul.restype = None
            lib.orc_matmul_at.argtypes = [i32, vp, i64, vp, vp, i64, vp, vp, vp, vp, vp]
            lib.orc_matmul_at.restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _t(type_) -> int:
    return TYPES[type_] if isinstance(type_, str) else int(type_)


def iq4nl_table() -> np.ndarray:
    """The oracle's own copy of the 16-entry IQ4_NL table (int8)."""
    lib = _load()
    arr = (ctypes.c_int8 * 16).in_dll(lib, "orc_iq4nl_table")
    return np.array(list(arr), dtype=np.int8)


def _lut(lut):
    return np.ascontiguousarray(iq4nl_table() if lut is None else np.asarray(lut, dtype=np.int8))


def f16_to_f32(h: int) -> float:
    return float(_load().orc_f16_to_f32(int(h) & 0xFFFF))


def f32_to_f16(x: float) -> int:
    return int(_load().orc_f32_to_f16(float(x)))


def e8m0_to_f16_bits(e: int) -> int:
    """The MXFP4 row scale as fp16 bits (the pages' clamp(e - 112, 0, 30) << 10)."""
    return int(_load().orc_e8m0_to_f16_bits(int(e)))


def block_bytes(type_) -> int:
    return int(_load().orc_block_bytes(_t(type_)))


def row_bytes(type_, K: int) -> int:
    """Bytes of one flat row of K weights (K/32 blocks, or K/256 Q4_K super-blocks)."""
    return int(_load().orc_row_bytes(_t(type_), K))


def _check_k(type_, K: int) -> None:
    assert K % 32 == 0 and (_t(type_) != Q4_K or K % 256 == 0), "K must be a multiple of the block length"


def tile_bytes(type_) -> int:
    return int(_load().orc_tile_bytes(_t(type_)))


def tile_index(ct: int, kt: int, n_k_tiles: int) -> int:
    return int(_load().orc_tile_index(ct, kt, n_k_tiles))


def tiled_bytes(type_, K: int, N: int) -> int:
    return int(_load().orc_tiled_bytes(_t(type_), K, N))


def quantize_block_q8_0(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (32,)
    q = np.zeros(32, np.int8)
    d = np.zeros(1, np.uint16)
    _load().orc_quantize_block_q8_0(_p(x), _p(q), _p(d))
    return q, int(d[0])


def quantize_rows(type_, w: np.ndarray, lut=None) -> np.ndarray:
    """fp32 [N, K] -> flat GGML blocks, uint8 [N, row_bytes(K)]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    _check_k(type_, K)
    out = np.zeros((N, row_bytes(type_, K)), np.uint8)
    lt = _lut(lut)
    _load().orc_quantize_rows(_t(type_), _p(w), N, K, _p(lt), _p(out))
    return out


def dequantize_flat(type_, flat: np.ndarray, N: int, K: int, lut=None) -> np.ndarray:
    flat = np.ascontiguousarray(flat, dtype=np.uint8)
    _check_k(type_, K)
    assert flat.size == N * row_bytes(type_, K)
    out = np.zeros((N, K), np.float64)
    lt = _lut(lut)
    _load().orc_dequantize_flat(_t(type_), _p(flat), N, K, _p(lt), _p(out))
    return out


def repack(type_, flat: np.ndarray, K: int, N: int) -> np.ndarray:
    flat = np.ascontiguousarray(flat, dtype=np.uint8)
    _check_k(type_, K)
    assert flat.size == N * row_bytes(type_, K)
    out = np.zeros(tiled_bytes(type_, K, N), np.uint8)
    _load().orc_repack(_t(type_), _p(flat), K, N, _p(out))
    return out


def unpack(type_, tiled: np.ndarray, K: int, N: int) -> np.ndarray:
    """Tiles -> flat rows for the block-32 types (a Q4_K tile holds rounded products of the
    super-block's fields, which cannot be split back)."""
    if _t(type_) == Q4_K:
        raise ValueError("Q4_K tiles cannot be unpacked")
    tiled = np.ascontiguousarray(tiled, dtype=np.uint8)
    assert tiled.size == tiled_bytes(type_, K, N)
    out = np.zeros((N, K // 32 * block_bytes(type_)), np.uint8)
    _load().orc_unpack(_t(type_), _p(tiled), K, N, _p(out))
    return out


def quantize_act(x: np.ndarray):
    """fp32 [M, K] -> (a_q int8 [M, K], a_d uint16 fp16 bits [M, K/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % 32 == 0
    a_q = np.zeros((M, K), np.int8)
    a_d = np.zeros((M, K // 32), np.uint16)
    _load().orc_quantize_act(_p(x), M, K, K, _p(a_q), _p(a_d))
    return a_q, a_d


def act_to_blocks(a_q: np.ndarray, a_d: np.ndarray) -> np.ndarray:
    """The activation arrays as GGML Q8_0 blocks: per row, K/32 blocks of {fp16 d; int8 qs[32]} (34 B).
    A byte rearrangement only; the library keeps the two arrays separate for aligned vector loads."""
    a_q = np.ascontiguousarray(a_q, dtype=np.int8)
    a_d = np.ascontiguousarray(a_d, dtype=np.uint16)
    M, K = a_q.shape
    out = np.zeros((M, K // 32, 34), np.uint8)
    out[:, :, 0:2] = a_d.astype("<u2").view(np.uint8).reshape(M, K // 32, 2)
    out[:, :, 2:] = a_q.view(np.uint8).reshape(M, K // 32, 32)
    return out.reshape(M, K // 32 * 34)


def blocks_to_act(blocks: np.ndarray, M: int, K: int):
    """Inverse of act_to_blocks: (a_q int8 [M, K], a_d uint16 [M, K/32])."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(M, K // 32, 34)
    a_d = np.ascontiguousarray(b[:, :, 0:2]).view("<u2").reshape(M, K // 32).astype(np.uint16)
    a_q = np.ascontiguousarray(b[:, :, 2:]).view(np.int8).reshape(M, K)
    return a_q, a_d


def matmul(type_, tiled: np.ndarray, K: int, N: int, a_q: np.ndarray, a_d: np.ndarray, lut=None):
    """Full output: (Y fp64 [M, N], B fp64 [M, N])."""
    tiled = np.ascontiguousarray(tiled, dtype=np.uint8)
    a_q = np.ascontiguousarray(a_q, dtype=np.int8)
    a_d = np.ascontiguousarray(a_d, dtype=np.uint16)
    M = a_q.shape[0]
    assert a_q.shape == (M, K) and a_d.shape == (M, K // 32)
    y = np.zeros((M, N), np.float64)
    b = np.zeros((M, N), np.float64)
    lt = _lut(lut)
    _load().orc_matmul(_t(type_), _p(tiled), K, N, _p(a_q), _p(a_d), M, _p(lt), _p(y), _p(b))
    return y, b


def matmul_at(type_, tiled: np.ndarray, K: int, a_q: np.ndarray, a_d: np.ndarray, ms, ns, lut=None):
    """Selected outputs Y[ms[i], ns[i]] and their bounds (fp64 vectors)."""
    tiled = np.ascontiguousarray(tiled, dtype=np.uint8)
    a_q = np.ascontiguousarray(a_q, dtype=np.int8)
    a_d = np.ascontiguousarray(a_d, dtype=np.uint16)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    assert ms.shape == ns.shape
    y = np.zeros(ms.size, np.float64)
    b = np.zeros(ms.size, np.float64)
    lt = _lut(lut)
    _load().orc_matmul_at(_t(type_), _p(tiled), K, _p(a_q), _p(a_d), ms.size, _p(ms), _p(ns), _p(lt),
                          _p(y), _p(b))
    return y, b

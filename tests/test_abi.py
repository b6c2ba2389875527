"""Host-side checks of libqmm that need no GPU: exported symbols, size queries, argument errors.

Every call below fails validation before anything is launched, so no CUDA device is touched.
"""
import ctypes
import os
import re

import pytest

import block_quantized_matmul_gb300 as qmm

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qmm.h")
INVALID, UNSUPPORTED, MISALIGNED = 1, 2, 3


@pytest.fixture(scope="module")
def L():
    from block_quantized_matmul_gb300 import build

    build.build()
    return qmm.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"QMM_API[^;(]*?\b(qmm_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_symbols()
    for required in ("qmm_repack", "qmm_quantize_act", "qmm_matmul", "qmm_tiled_size", "qmm_tile_size",
                     "qmm_status_str", "qmm_unpack"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_sizes(L):
    assert qmm.tile_size("q4_0") == 576 and qmm.tile_size("iq4_nl") == 576 and qmm.tile_size("q8_0") == 1088
    assert qmm.block_size("q4_0") == 18 and qmm.block_size("q8_0") == 34
    assert qmm.tiled_size("q4_0", 4096, 4096) == 9437184
    assert qmm.tiled_size("q8_0", 4096, 14336) == 62390272
    assert qmm.tiled_size("q8_0", 4096, 128256) == 558170112
    assert qmm.tiled_size("q4_0", 64, 33) == 4 * 576
    assert qmm.flat_size("q8_0", 64, 33) == 33 * 2 * 34
    assert qmm.tiled_size("q4_0", 33, 64) == 0 and qmm.tiled_size("q4_0", 0, 64) == 0
    assert qmm.tiled_size("q4_0", 64, 0) == 0 and qmm.tiled_size(7, 64, 64) == 0
    assert L.qmm_tile_size(9) == 0
    assert qmm.decode_max_m() >= 8
    # MXFP4: 544-byte tiles of 32 rows x 17-byte blocks
    assert qmm.tile_size("mxfp4") == 544 and qmm.block_size("mxfp4") == 17
    assert qmm.tiled_size("mxfp4", 4096, 14336) == 448 * 128 * 544
    assert qmm.flat_size("mxfp4", 64, 33) == 33 * 2 * 17
    # Q4_1: 640-byte tiles of 32 rows x 20-byte blocks
    assert qmm.tile_size("q4_1") == 640 and qmm.block_size("q4_1") == 20
    assert qmm.tiled_size("q4_1", 4096, 4096) == 128 * 128 * 640


def test_mxfp4_flat_blocks_need_no_alignment(L):
    # 17-byte blocks are read byte by byte: an odd flat pointer is accepted for MXFP4 (the call then
    # fails only on the too-large K, before any launch), but not for the 18-byte formats
    assert L.qmm_repack(3, P + 1, 48, 64, P, None) == INVALID
    assert L.qmm_repack(0, P + 1, 64, 64, P, None) == MISALIGNED
    assert L.qmm_repack(3, P, 64, 64, P + 8, None) == MISALIGNED


def test_iq4nl_table_matches_the_oracle(L, orc):
    assert qmm.iq4nl_table() == list(orc.iq4nl_table())


def test_status_strings(L):
    for st in range(8):
        assert L.qmm_status_str(st)
    assert L.qmm_status_str(7) != L.qmm_status_str(99)
    assert L.qmm_status_str(99) == b"unknown status"


P = 1 << 20          # a fake, 16-byte aligned, non-null address (never dereferenced: validation fails first)


@pytest.mark.parametrize("args,expect", [
    ((0, P, 0, 64, P, P, 1, P, 64, None), INVALID),      # K = 0
    ((0, P, 48, 64, P, P, 1, P, 64, None), INVALID),     # K % 32
    ((0, P, 64, 0, P, P, 1, P, 64, None), INVALID),      # N = 0
    ((0, P, 64, 64, P, P, 0, P, 64, None), INVALID),     # M = 0
    ((0, P, 64, 64, P, P, -3, P, 64, None), INVALID),    # M < 0
    ((0, P, 64, 64, P, P, 1, P, 63, None), INVALID),     # ldy < N
    ((0, None, 64, 64, P, P, 1, P, 64, None), INVALID),  # NULL weight
    ((0, P, 64, 64, None, P, 1, P, 64, None), INVALID),  # NULL a_q
    ((0, P, 64, 64, P, None, 1, P, 64, None), INVALID),  # NULL a_d
    ((0, P, 64, 64, P, P, 1, None, 64, None), INVALID),  # NULL y
    ((99, P, 64, 64, P, P, 1, P, 64, None), UNSUPPORTED),  # unknown type
    ((0, P + 8, 64, 64, P, P, 1, P, 64, None), MISALIGNED),
    ((0, P, 64, 64, P + 4, P, 1, P, 64, None), MISALIGNED),
    ((0, P, 64, 64, P, P + 2, 1, P, 64, None), MISALIGNED),
    ((0, P, 64, 64, P, P, 1, P + 2, 64, None), MISALIGNED),
])
def test_matmul_argument_errors(L, args, expect):
    assert L.qmm_matmul(*args) == expect


def test_matmul_path_rejects_unknown_path(L):
    assert L.qmm_matmul_path(0, P, 64, 64, P, P, 1, P, 64, 7, None) == UNSUPPORTED


def test_quantize_act_argument_errors(L):
    assert L.qmm_quantize_act(P, 0, 64, 64, P, P, None) == INVALID
    assert L.qmm_quantize_act(P, 2, 40, 64, P, P, None) == INVALID
    assert L.qmm_quantize_act(P, 2, 64, 32, P, P, None) == INVALID
    assert L.qmm_quantize_act(None, 2, 64, 64, P, P, None) == INVALID
    assert L.qmm_quantize_act(P + 1, 2, 64, 64, P, P, None) == MISALIGNED
    assert L.qmm_quantize_act(P, 2, 64, 64, P + 4, P, None) == MISALIGNED
    assert L.qmm_quantize_act(P, 2, 64, 64, P, P + 2, None) == MISALIGNED


def test_repack_and_quantize_weight_argument_errors(L):
    assert L.qmm_repack(0, P, 48, 64, P, None) == INVALID
    assert L.qmm_repack(0, None, 64, 64, P, None) == INVALID
    assert L.qmm_repack(99, P, 64, 64, P, None) == UNSUPPORTED
    assert L.qmm_repack(0, P + 1, 64, 64, P, None) == MISALIGNED
    assert L.qmm_repack(0, P, 64, 64, P + 8, None) == MISALIGNED
    assert L.qmm_unpack(1, P + 8, 64, 64, P, None) == MISALIGNED
    assert L.qmm_unpack(1, P, 64, -1, P, None) == INVALID
    assert L.qmm_quantize_weight(0, P, 64, 64, 60, P, None) == INVALID      # ldw < K
    assert L.qmm_quantize_weight(0, P, 64, 64, 66, P, None) == MISALIGNED   # ldw % 4
    assert L.qmm_quantize_weight(0, P + 4, 64, 64, 64, P, None) == MISALIGNED
    assert L.qmm_quantize_weight(99, P, 64, 64, 64, P, None) == UNSUPPORTED


def test_binding_raises_on_error(L):
    with pytest.raises(qmm.QmmError):
        qmm.qmm_matmul("q4_0", P, 48, 64, P, P, 1, P, 64, stream=0)


def test_matmul_ws_argument_errors(L):
    need = L.qmm_matmul_workspace_size(64, 256)
    assert need >= 64 * 256 * 2
    assert L.qmm_matmul_workspace_size(0, 256) == 0 and L.qmm_matmul_workspace_size(64, 48) == 0
    # M > 16 takes the GEMM path, which needs the workspace
    assert L.qmm_matmul_ws(0, P, 256, 64, P, P, 64, P, 64, None, need, None) == INVALID
    assert L.qmm_matmul_ws(0, P, 256, 64, P, P, 64, P, 64, P, need - 1, None) == INVALID
    assert L.qmm_matmul_ws(0, P, 256, 64, P, P, 64, P, 64, P + 16, need, None) == MISALIGNED
    assert L.qmm_matmul_ws(0, P, 48, 64, P, P, 64, P, 64, P, need, None) == INVALID


def test_workspace_sizes_as_documented(L):
    # the folded-scale GEMM's token operand is two fp16 terms per element (4 B), plus the block-scale
    # and per-row regions of the exact-integer GEMM: about 4.2 B per activation element
    for M, K in [(17, 32), (300, 1024), (512, 4096)]:
        need = L.qmm_matmul_workspace_size(M, K)
        assert 4 * M * K <= need <= 4.3 * M * K + 4096, (M, K, need)
    # the no-allocation scratch: 16 MiB, which holds M = 960 tokens at K = 4096 but not 1024
    limit = L.qmm_matmul_noalloc_max_workspace()
    assert limit == 16 << 20
    assert L.qmm_matmul_workspace_size(960, 4096) <= limit < L.qmm_matmul_workspace_size(1024, 4096)


def test_matmul_f32_argument_errors(L):
    f = L.qmm_matmul_f32
    assert f(0, P, 48, 64, P, 64, 1, P, 64, None) == INVALID     # K % 32
    assert f(0, P, 64, 64, P, 63, 1, P, 64, None) == INVALID     # ldx < K
    assert f(0, P, 64, 64, P, 64, 0, P, 64, None) == INVALID     # M = 0
    assert f(0, P, 64, 64, P, 64, 1, P, 63, None) == INVALID     # ldy < N
    assert f(0, None, 64, 64, P, 64, 1, P, 64, None) == INVALID  # NULL weight
    assert f(0, P, 64, 64, None, 64, 1, P, 64, None) == INVALID  # NULL x
    assert f(0, P, 64, 64, P, 64, 1, None, 64, None) == INVALID  # NULL y
    assert f(99, P, 64, 64, P, 64, 1, P, 64, None) == UNSUPPORTED
    assert f(0, P + 8, 64, 64, P, 64, 1, P, 64, None) == MISALIGNED
    assert f(0, P, 64, 64, P + 2, 64, 1, P, 64, None) == MISALIGNED
    assert f(0, P, 64, 64, P, 64, 1, P + 1, 64, None) == MISALIGNED


def test_matmul_f32_ws_argument_errors(L):
    assert L.qmm_matmul_f32_workspace_size(4, 4096) == 4 * 4096 * 4
    assert L.qmm_matmul_f32_workspace_size(3, 32) == 512          # 384 B rounded up to 256
    assert L.qmm_matmul_f32_workspace_size(0, 64) == 0 and L.qmm_matmul_f32_workspace_size(1, 48) == 0
    need = L.qmm_matmul_f32_workspace_size(1, 64)
    f = L.qmm_matmul_f32_ws
    # the arguments of qmm_matmul_f32 are checked first
    assert f(0, P, 48, 64, P, 64, 1, P, 64, P, need, None) == INVALID
    assert f(0, P, 64, 64, P, 63, 1, P, 64, P, need, None) == INVALID
    assert f(0, P, 64, 64, P + 2, 64, 1, P, 64, P, need, None) == MISALIGNED
    # then the workspace
    assert f(0, P, 64, 64, P, 64, 1, P, 64, None, need, None) == INVALID
    assert f(0, P, 64, 64, P, 64, 1, P, 64, P, need - 1, None) == INVALID
    assert f(0, P, 64, 64, P, 64, 1, P, 64, P + 16, need, None) == MISALIGNED


def test_matmul_flat_argument_errors(L):
    f = L.qmm_matmul_flat
    assert f(0, P, 48, 64, P, P, 1, P, 64, None) == INVALID       # K % 32
    assert f(0, P, 512, 64, P, P, 0, P, 64, None) == INVALID      # M = 0
    assert f(0, P, 512, 64, P, P, 1, P, 63, None) == INVALID      # ldy < N
    assert f(0, None, 512, 64, P, P, 1, P, 64, None) == INVALID   # NULL weight
    assert f(99, P, 512, 64, P, P, 1, P, 64, None) == UNSUPPORTED
    assert f(0, P + 8, 512, 64, P, P, 1, P, 64, None) == MISALIGNED
    # a flat row must be a whole number of 16-byte units: 2 Q4_0 blocks = 36 B, 4 Q8_0 blocks = 136 B,
    # 8 MXFP4 blocks = 136 B
    assert f(0, P, 64, 64, P, P, 1, P, 64, None) == UNSUPPORTED
    assert f(1, P, 128, 64, P, P, 1, P, 64, None) == UNSUPPORTED
    assert f(3, P, 256, 64, P, P, 1, P, 64, None) == UNSUPPORTED


def test_q4_k_sizes_and_argument_errors(L):
    assert qmm.block_size("q4_k") == 144 and qmm.tile_size("q4_k") == 640
    assert qmm.flat_size("q4_k", 4096, 10) == 10 * 16 * 144
    assert qmm.tiled_size("q4_k", 4096, 10) == 128 * 640
    assert qmm.flat_size("q4_k", 288, 10) == 0 and qmm.tiled_size("q4_k", 288, 10) == 0   # K % 256
    assert L.qmm_quantize_weight(5, P, 4, 288, 288, P, None) == INVALID
    assert L.qmm_repack(5, P, 288, 4, P, None) == INVALID
    assert L.qmm_repack(5, P + 2, 256, 4, P, None) == MISALIGNED          # super-blocks are read as words
    assert L.qmm_unpack(5, P, 256, 4, P, None) == UNSUPPORTED             # tiles hold rounded products
    assert L.qmm_matmul(5, P, 288, 64, P, P, 1, P, 64, None) == INVALID
    assert L.qmm_matmul_f32(5, P, 288, 64, P, 288, 1, P, 64, None) == INVALID
    assert L.qmm_matmul_flat(5, P, 288, 64, P, P, 1, P, 64, None) == INVALID


def test_selftest_timeout_argument_errors(L):
    f = L.qmm_selftest_timeout
    assert f(3, 100_000_000, P, None) == INVALID              # unit
    assert f(-1, 100_000_000, P, None) == INVALID
    assert f(0, 999_999, P, None) == INVALID                  # below 1 ms
    assert f(1, 2_000_000_001, P, None) == INVALID            # above 2 s
    assert f(0, 100_000_000, None, None) == INVALID
    assert f(0, 100_000_000, P + 2, None) == MISALIGNED


def test_product_calls_cap_k(L):
    # the fp32 accumulation bound of every kernel is derived up to K = 131072 (4096 blocks); longer
    # rows are refused before anything is launched
    K = 131072 + 32
    assert L.qmm_matmul(1, P, K, 64, P, P, 1, P, 64, None) == INVALID
    assert L.qmm_matmul_path(1, P, K, 64, P, P, 300, P, 64, 2, None) == INVALID
    assert L.qmm_matmul_ws(1, P, K, 64, P, P, 300, P, 64, P, 1 << 40, None) == INVALID
    assert L.qmm_matmul_noalloc(1, P, K, 64, P, P, 300, P, 64, None) == INVALID
    assert L.qmm_matmul_f32(1, P, K, 64, P, K, 1, P, 64, None) == INVALID
    assert L.qmm_matmul_flat(1, P, K, 64, P, P, 1, P, 64, None) == INVALID
    # the weight-side calls are not products and keep the wider limit
    assert L.qmm_tiled_size(1, K, 64) > 0


def test_debug_build_is_a_separate_library_with_the_checks_on(monkeypatch, tmp_path):
    """build(debug=True) compiles every source with -DQMM_DEBUG into its own object folder and links
    libqmm_debug.so; the release build passes no such flag (nothing is compiled here: nvcc is faked)."""
    from block_quantized_matmul_gb300 import build

    calls = []

    class Done:
        returncode = 0
        stdout = stderr = ""

    def fake_run(cmd, capture_output=True, text=True):
        calls.append(cmd)
        out = cmd[cmd.index("-o") + 1]
        os.makedirs(os.path.dirname(out), exist_ok=True)
        with open(out, "w") as f:
            f.write("")
        return Done()

    monkeypatch.setattr(build.subprocess, "run", fake_run)
    monkeypatch.setattr(build, "OBJ_DIR", str(tmp_path / "_build"))
    monkeypatch.setattr(build, "LIB", str(tmp_path / "libqmm.so"))
    monkeypatch.setattr(build, "LIB_DEBUG", str(tmp_path / "libqmm_debug.so"))
    assert build.build(force=True, debug=True) == str(tmp_path / "libqmm_debug.so")
    compiles = [c for c in calls if "-c" in c]
    assert compiles and all("-DQMM_DEBUG" in c for c in compiles)
    assert all(os.path.dirname(c[c.index("-o") + 1]).endswith("_build_debug") for c in compiles)
    calls.clear()
    assert build.build(force=True, debug=False) == str(tmp_path / "libqmm.so")
    assert not any("-DQMM_DEBUG" in c for c in calls)
    # the environment switch selects the debug build by default
    monkeypatch.setenv("QMM_DEBUG", "1")
    calls.clear()
    assert build.build(force=True) == str(tmp_path / "libqmm_debug.so")


def test_bounds_status_is_documented(L):
    assert L.qmm_status_str(7) == b"device bounds check failed (debug build)"
    with open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qmm.h")) as f:
        assert "QMM_ERR_BOUNDS = 7" in f.read()

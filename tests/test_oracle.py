"""Pins for the CPU oracle: each test checks it against something other than itself.

Sources: "Hexagon backend developer details", section "Tiled Weight Formats" ("Tile Dimensions and
Grid Layout", "Block-32 Quantized Formats").  Fixtures under tests/golden/ were worked out by hand
from those sections.
"""
import os

import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TYPES = ["q4_0", "q8_0", "iq4_nl", "mxfp4", "q4_1"]


# ---------------------------------------------------------------------------------------------
# binary16 conversion: against numpy's IEEE float16 (an independent library routine)
# ---------------------------------------------------------------------------------------------
def test_f16_conversion_matches_numpy(orc):
    rng = np.random.default_rng(123)
    vals = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 3000),
        np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.0, 65520.0, 1e9, -1e9, 6.1035156e-05, 6.0e-08,
                  5.9604645e-08, 2.9802322e-08, 2.98023259e-08, 1e-40, 0.5 + 2.0 ** -12,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2048.0 + 1.0, 2048.0 + 3.0], dtype=np.float32),
    ])
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.array([v], dtype=np.float32).astype(np.float16).view(np.uint16)[0])
        got = orc.f32_to_f16(float(v))
        assert got == want, (float(v), hex(got), hex(want))
    for h in list(range(0, 0x7C00, 7)) + [0x0001, 0x03FF, 0x0400, 0x7BFF, 0x7C00, 0x8001, 0xFBFF, 0xFC00]:
        want = float(np.array([h], dtype=np.uint16).view(np.float16).astype(np.float32)[0])
        assert orc.f16_to_f32(h) == want, hex(h)


# ---------------------------------------------------------------------------------------------
# sizes and the tile grid
# ---------------------------------------------------------------------------------------------
def test_tile_and_block_sizes(orc):
    # Tile sizes are printed on the pages; the flat blocks are 18 / 34 bytes, so tiling is lossless.
    assert orc.tile_bytes("q4_0") == 576 and orc.tile_bytes("iq4_nl") == 576
    assert orc.tile_bytes("q8_0") == 1088
    assert 32 * orc.block_bytes("q4_0") == 576 and 32 * orc.block_bytes("iq4_nl") == 576
    assert 32 * orc.block_bytes("q8_0") == 1088
    assert orc.tile_bytes("mxfp4") == 544 and 32 * orc.block_bytes("mxfp4") == 544
    assert orc.tile_bytes("q4_1") == 640 and 32 * orc.block_bytes("q4_1") == 640


@pytest.mark.parametrize("K,N,type_,tiles", [
    (4096, 4096, "q4_0", 128 * 128),
    (4096, 14336, "q8_0", 448 * 128),
    (4096, 128256, "q8_0", 4008 * 128),
    (64, 33, "q4_0", 2 * 2),        # 33 rows -> 2 column tiles (ceil), 2 K tiles
    (32, 1, "iq4_nl", 1),
])
def test_tiled_size_grid(orc, K, N, type_, tiles):
    assert orc.tiled_bytes(type_, K, N) == tiles * orc.tile_bytes(type_)


def test_tile_index_order(orc):
    # tile_idx = ct * n_k_tiles + kt: the K-tiles of one column tile are consecutive.
    assert orc.tile_index(0, 0, 128) == 0
    assert orc.tile_index(0, 127, 128) == 127
    assert orc.tile_index(1, 0, 128) == 128
    assert orc.tile_index(3, 5, 7) == 26


# ---------------------------------------------------------------------------------------------
# repack: hand-placed quants land where the pages say
# ---------------------------------------------------------------------------------------------
def _read_positions():
    rows = []
    with open(os.path.join(GOLDEN, "tile_positions.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b, c = [p.split() for p in line.split("|")]
            rows.append((a[0], int(a[1]), int(a[2]), int(a[3]), int(b[0]), int(b[1]), int(c[0]),
                         int(c[1]), int(c[2])))
    return rows


@pytest.mark.parametrize("case", _read_positions())
def test_one_hot_tile_position(orc, case):
    type_, row, col, code, fbyte, fshift, tbyte, tshift, sbyte = case
    bb, ts = orc.block_bytes(type_), orc.tile_bytes(type_)
    N, K = 32, 32
    flat = np.zeros((N, bb), np.uint8)
    raw = code & 0xFF if type_ == "q8_0" else code << fshift
    flat[row, fbyte] = raw
    expect = np.zeros(ts, np.uint8)
    if type_ == "mxfp4":
        flat[row, 0] = 0x7B                    # E8M0 exponent byte of that row
        expect[sbyte] = 0x7B
    elif type_ == "q4_1":
        flat[row, 0:4] = (0x34, 0x12, 0x78, 0x56)    # fp16 d = 0x1234, m = 0x5678 on that row
        expect[sbyte:sbyte + 4] = (0x34, 0x12, 0x78, 0x56)
    else:
        flat[row, 0:2] = (0x34, 0x12)          # fp16 scale bits 0x1234 on that row
        expect[sbyte], expect[sbyte + 1] = 0x34, 0x12
    tiled = orc.repack(type_, flat, K, N)
    assert tiled.size == ts
    expect[tbyte] = (code & 0xFF) if type_ == "q8_0" else (code << tshift)
    assert np.array_equal(tiled, expect), np.nonzero(tiled != expect)


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("K,N", [(32, 1), (64, 33), (96, 64), (128, 100)])
def test_repack_unpack_roundtrip_and_padding(orc, type_, K, N):
    rng = np.random.default_rng(K * 1000 + N)
    flat = rng.integers(0, 256, size=(N, K // 32 * orc.block_bytes(type_)), dtype=np.uint8)
    tiled = orc.repack(type_, flat, K, N)
    assert np.array_equal(orc.unpack(type_, tiled, K, N), flat)
    # rows past N in the last column tile are zero bytes
    ts, nkt = orc.tile_bytes(type_), K // 32
    last_ct = (N + 31) // 32 - 1
    pad_rows = [r for r in range(32) if last_ct * 32 + r >= N]
    if pad_rows:
        for kt in range(nkt):
            t = tiled[(last_ct * nkt + kt) * ts:(last_ct * nkt + kt + 1) * ts]
            for r in pad_rows:
                if type_ == "q8_0":
                    assert all(t[cp * 64 + 2 * r + h] == 0 for cp in range(16) for h in range(2))
                    assert t[1024 + 2 * r] == 0 and t[1025 + 2 * r] == 0
                elif type_ == "mxfp4":
                    assert all(t[cp * 32 + r] == 0 for cp in range(16))
                    assert t[512 + r] == 0
                elif type_ == "q4_1":
                    assert all(t[cp * 32 + r] == 0 for cp in range(16))
                    assert not t[512 + 4 * r:516 + 4 * r].any()
                else:
                    assert all(t[cp * 32 + r] == 0 for cp in range(16))
                    assert t[512 + 2 * r] == 0 and t[513 + 2 * r] == 0


def test_repack_keeps_k_tiles_of_a_column_tile_contiguous(orc):
    # Block kt of row n must land in tile ct*n_k_tiles + kt: mark each block by its scale.
    K, N = 32 * 5, 64
    bb, ts = orc.block_bytes("q8_0"), orc.tile_bytes("q8_0")
    flat = np.zeros((N, 5 * bb), np.uint8)
    for n in range(N):
        for kt in range(5):
            flat[n, kt * bb] = n
            flat[n, kt * bb + 1] = kt
    tiled = orc.repack("q8_0", flat, K, N)
    for ct in range(2):
        for kt in range(5):
            t = tiled[(ct * 5 + kt) * ts:(ct * 5 + kt + 1) * ts]
            for r in range(32):
                assert t[1024 + 2 * r] == ct * 32 + r and t[1025 + 2 * r] == kt


# ---------------------------------------------------------------------------------------------
# activation quantization
# ---------------------------------------------------------------------------------------------
def _read_act_cases():
    cases = []
    with open(os.path.join(GOLDEN, "act_quant_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, xs, qs, d = [p.strip() for p in line.split("|")]
            x = np.zeros(32, np.float32)
            q = np.zeros(32, np.int8)
            for tok in xs.split():
                i, v = tok.split(":")
                x[int(i)] = np.float32(float(v))
            for tok in qs.split():
                i, v = tok.split(":")
                q[int(i)] = int(v)
            cases.append((name, x, q, int(d, 16)))
    return cases


@pytest.mark.parametrize("case", _read_act_cases(), ids=lambda c: c[0])
def test_act_quant_hand_cases(orc, case):
    _, x, q, d16 = case
    got_q, got_d = orc.quantize_block_q8_0(x)
    assert np.array_equal(got_q, q)
    assert got_d == d16


def test_act_quant_invariants(orc):
    x = synth.activations(16, 4096, outliers=True)
    a_q, a_d = orc.quantize_act(x)
    assert np.abs(a_q.astype(np.int32)).max() <= 127
    blocks = x.reshape(16, 128, 32)
    amax_idx = np.abs(blocks).argmax(axis=2)
    qb = a_q.reshape(16, 128, 32)
    picked = np.take_along_axis(qb, amax_idx[..., None], axis=2)[..., 0]
    assert np.all(np.abs(picked.astype(np.int32)) == 127)          # the largest element maps to +-127
    # dequantized activations stay within half a step (plus the fp16 scale rounding) of x
    d = a_d.view(np.float16).astype(np.float64)[..., None]
    err = np.abs(qb * d - blocks)
    assert np.all(err <= d * (0.5 + 127 * 2.0 ** -11) + 1e-30)


# ---------------------------------------------------------------------------------------------
# weight quantizers (test-data generators)
# ---------------------------------------------------------------------------------------------
def test_q4_0_hand_case(orc):
    x = np.zeros((1, 32), np.float32)
    x[0, :4] = [-1.6, 0.2, 0.0, 1.0]
    flat = orc.quantize_rows("q4_0", x)
    d = np.array([int(flat[0, 0]) | (int(flat[0, 1]) << 8)], np.uint16).view(np.float16)[0]
    assert d == np.float16(0.2)
    codes = [(flat[0, 2 + j] & 15) if j < 16 else (flat[0, 2 + j - 16] >> 4) for j in range(32)]
    assert codes[:4] == [0, 9, 8, 13]
    assert all(c == 8 for c in codes[4:])


def test_q4_0_tie_takes_the_first_extreme(orc):
    """|0.5| = |-0.5|: the first element sets the sign, d = 0.5/-8 = -0.0625 (1/d = -16), so 0.5 maps
    to trunc(-8 + 8.5) = 0, -0.5 to min(15, trunc(16.5)) = 15 and 0 to 8 (worked by hand)."""
    x = np.zeros((1, 32), np.float32)
    x[0, :2] = [0.5, -0.5]
    flat = orc.quantize_rows("q4_0", x)
    d = np.array([int(flat[0, 0]) | (int(flat[0, 1]) << 8)], np.uint16).view(np.float16)[0]
    assert d == np.float16(-0.0625)
    codes = [(flat[0, 2 + j] & 15) if j < 16 else (flat[0, 2 + j - 16] >> 4) for j in range(32)]
    assert codes[:3] == [0, 15, 8]


@pytest.mark.parametrize("type_", TYPES)
def test_weight_quantizer_error_bound(orc, type_):
    w = synth.weights(64, 256)
    flat = orc.quantize_rows(type_, w)
    deq = orc.dequantize_flat(type_, flat, 64, 256)
    blocks = w.reshape(64, 8, 32).astype(np.float64)
    dq = deq.reshape(64, 8, 32)
    amax = np.abs(blocks).max(axis=2, keepdims=True)
    if type_ == "q8_0":
        step = amax / 127
        assert np.all(np.abs(dq - blocks) <= step * (0.5 + 127 * 2.0 ** -11) + 1e-12)
    elif type_ == "q4_0":
        step = amax / 8
        assert np.all(np.abs(dq - blocks) <= step * (1.0 + 8 * 2.0 ** -11) + 1e-12)
    elif type_ == "q4_1":
        # affine: step (max - min)/15, rounding to nearest (<= step/2) plus the fp16 roundings of d and m
        mn = blocks.min(axis=2, keepdims=True)
        mx = blocks.max(axis=2, keepdims=True)
        step = (mx - mn) / 15
        assert np.all(np.abs(dq - blocks) <= step * (0.5 + 16 * 2.0 ** -11) + np.abs(mn) * 2.0 ** -11 + 1e-12)
    elif type_ == "mxfp4":
        # scale 2^(floor(log2 amax) - 2): levels up to 6 * scale cover amax < 8 * scale except the top
        # (saturation at 6 * scale); the widest gap below 6 is 2 * scale (between 4 and 6)
        scale = 2.0 ** (np.floor(np.log2(amax)) - 2)
        err = np.abs(dq - blocks)
        assert np.all(err <= np.maximum(scale, amax - 6 * scale) + 1e-12)
    else:
        # d = m / lut[0] puts the block's extreme m exactly on lut[0] (d > 0 for a negative m, d < 0 for
        # a positive one).  Inside the levels the error is at most half the widest gap; past the other
        # end of the (asymmetric) table, x can reach |m| while the last level is |d| * |lut[15]|.
        lut = orc.iq4nl_table().astype(np.float64)
        step = amax / 127
        reach = max(np.diff(lut).max() / 2, 127 - abs(lut[-1]))
        assert np.all(np.abs(dq - blocks) <= step * (reach + 127 * 2.0 ** -11) + 1e-12)


def test_iq4_nl_picks_nearest_entry(orc):
    # Brute force in the precision the rule is stated in (fp32): no other entry is strictly closer.
    w = synth.weights(8, 128)
    lut = orc.iq4nl_table()
    flat = orc.quantize_rows("iq4_nl", w)
    for n in range(8):
        for b in range(4):
            blk = flat[n, b * 18:(b + 1) * 18]
            d = np.float32(np.array([int(blk[0]) | (int(blk[1]) << 8)], np.uint16).view(np.float16)[0])
            levels = (d * lut.astype(np.float32)).astype(np.float32)
            for j in range(32):
                c = (blk[2 + j] & 15) if j < 16 else (blk[2 + j - 16] >> 4)
                x = w[n, b * 32 + j]
                errs = np.abs(np.float32(x) - levels)
                assert errs[c] <= errs.min()
                assert c == int(np.argmax(errs == errs.min()))     # lowest index among ties


def test_iq4_nl_table_is_ggmls_published_table(orc):
    # The pages name the table (iq4_nl_to_fp16_lut) but print no values.  The oracle holds the 16
    # levels of GGML's published IQ4_NL format, written out here from that format's definition.
    ggml_iq4_nl = [-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113]
    table = orc.iq4nl_table()
    assert table.dtype == np.int8 and table.shape == (16,)
    assert table.tolist() == ggml_iq4_nl
    # what the kernels rely on: ascending, lut[0] the most negative level, every |level| <= 127
    assert np.all(np.diff(table.astype(int)) > 0) and table[0] == -127 and np.abs(table.astype(int)).max() == 127


# ---------------------------------------------------------------------------------------------
# matmul: fp64 brute force on the FLAT blocks (never touches the tile layout) vs the tiled oracle
# ---------------------------------------------------------------------------------------------
def _brute(orc, type_, flat, a_q, a_d, N, K, lut=None):
    W = orc.dequantize_flat(type_, flat, N, K, lut)                        # [N, K] fp64
    A = a_q.astype(np.float64) * np.repeat(a_d.view(np.float16).astype(np.float64), 32, axis=1)
    return A @ W.T


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("K,N,M", [(32, 1, 1), (64, 31, 3), (96, 32, 1), (96, 33, 3), (160, 65, 2)])
def test_matmul_matches_fp64_brute_force(orc, type_, K, N, M):
    w = synth.weights(N, K, seed=K + N)
    x = synth.activations(M, K, seed=M + 7, outliers=True)
    flat = orc.quantize_rows(type_, w)
    tiled = orc.repack(type_, flat, K, N)
    a_q, a_d = orc.quantize_act(x)
    y, bound = orc.matmul(type_, tiled, K, N, a_q, a_d)
    ref = _brute(orc, type_, flat, a_q, a_d, N, K)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)
    assert np.all(bound >= np.abs(y) - 1e-15)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ys, bs = orc.matmul_at(type_, tiled, K, a_q, a_d, ms.ravel(), ns.ravel())
    assert np.array_equal(ys, y.ravel()) and np.array_equal(bs, bound.ravel())


def test_matmul_one_hot_activation_reads_weight_column(orc):
    K, N = 64, 40
    w = synth.weights(N, K, seed=5)
    flat = orc.quantize_rows("q4_0", w)
    tiled = orc.repack("q4_0", flat, K, N)
    W = orc.dequantize_flat("q4_0", flat, N, K)
    for k in (0, 13, 33, 63):
        a_q = np.zeros((1, K), np.int8)
        a_q[0, k] = 1
        a_d = np.full((1, K // 32), np.float16(1.0).view(np.uint16), np.uint16)
        y, _ = orc.matmul("q4_0", tiled, K, N, a_q, a_d)
        assert np.array_equal(y[0], W[:, k])


def test_matmul_zero_and_linearity(orc):
    K, N, M = 96, 48, 2
    rng = np.random.default_rng(9)
    flat = orc.quantize_rows("q8_0", synth.weights(N, K, seed=3))
    tiled = orc.repack("q8_0", flat, K, N)
    a_d = synth.activations(M, K // 32, seed=4).astype(np.float16).view(np.uint16)
    q1 = rng.integers(-60, 60, size=(M, K), dtype=np.int8)
    q2 = rng.integers(-60, 60, size=(M, K), dtype=np.int8)
    y1, _ = orc.matmul("q8_0", tiled, K, N, q1, a_d)
    y2, _ = orc.matmul("q8_0", tiled, K, N, q2, a_d)
    y12, _ = orc.matmul("q8_0", tiled, K, N, (q1 + q2).astype(np.int8), a_d)
    assert np.allclose(y12, y1 + y2, rtol=1e-13, atol=1e-15)
    y0, b0 = orc.matmul("q8_0", tiled, K, N, np.zeros((M, K), np.int8), a_d)
    assert not y0.any() and not b0.any()


def test_iq4_nl_with_offset_table_equals_q4_0(orc):
    # With lut[i] = i - 8 the IQ4_NL dequantization is the Q4_0 one on the same bytes.
    K, N, M = 128, 64, 3
    flat = orc.quantize_rows("q4_0", synth.weights(N, K, seed=11))
    tiled = orc.repack("q4_0", flat, K, N)
    a_q, a_d = orc.quantize_act(synth.activations(M, K, seed=12))
    y4, b4 = orc.matmul("q4_0", tiled, K, N, a_q, a_d)
    yi, bi = orc.matmul("iq4_nl", tiled, K, N, a_q, a_d, lut=np.arange(16) - 8)
    assert np.array_equal(y4, yi) and np.array_equal(b4, bi)


# ---------------------------------------------------------------------------------------------
# MXFP4: the pages' E8M0 conversion and the OCP E2M1 code set
# ---------------------------------------------------------------------------------------------
# OCP Microscaling FP4 (E2M1) values of codes 0..7; codes 8..15 are their negatives (sign bit 3).
OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e8m0_scale_follows_the_pages_formula(orc):
    # "clamp(e - 112, 0, 30) << 10" read as fp16 bits: 2^(e-127) in 113..142, 0 below, 2^15 above.
    for e in range(256):
        v = float(np.array([orc.e8m0_to_f16_bits(e)], np.uint16).view(np.float16)[0])
        if e <= 112:
            assert v == 0.0
        elif e <= 142:
            assert v == 2.0 ** (e - 127)
        else:
            assert v == 2.0 ** 15
    assert orc.e8m0_to_f16_bits(127) == 0x3C00          # 1.0


def test_mxfp4_dequant_is_e2m1_times_scale(orc):
    # Every code at several exponents, decoded from the raw bytes with the OCP table and numpy fp16.
    flat = np.zeros((16, 17), np.uint8)
    for r in range(16):
        flat[r, 0] = 100 + 3 * r                          # exponents 100..145 (some flushed, some clamped)
        for j in range(32):
            code = (j + r) % 16
            if j < 16:
                flat[r, 1 + j] |= code
            else:
                flat[r, 1 + j - 16] |= code << 4
    deq = orc.dequantize_flat("mxfp4", flat, 16, 32)
    for r in range(16):
        e = int(flat[r, 0])
        s = float(np.array([min(max(e - 112, 0), 30) << 10], np.uint16).view(np.float16)[0])
        for j in range(32):
            code = (j + r) % 16
            v = OCP_E2M1[code & 7] * (-1.0 if code & 8 else 1.0)
            assert deq[r, j] == v * s, (r, j, code, e)


def test_mxfp4_quantizer_exact_values_and_nearest_level(orc):
    rng = np.random.default_rng(5)
    # exactly representable blocks come back unchanged (the largest magnitude 6 * 2^k fixes e)
    levels = np.array(OCP_E2M1 + [-v for v in OCP_E2M1], np.float32)
    w = np.stack([np.float32(2.0 ** k) * np.concatenate([[np.float32(6.0)], rng.choice(levels, 31)]).astype(np.float32)
                  for k in range(-6, 7)]).astype(np.float32)
    flat = orc.quantize_rows("mxfp4", w)
    assert np.array_equal(orc.dequantize_flat("mxfp4", flat, w.shape[0], 32), w.astype(np.float64))
    # otherwise each element takes a nearest level of its block's scale (lowest code on ties)
    w = synth.weights(8, 64)
    flat = orc.quantize_rows("mxfp4", w)
    for n in range(8):
        for b in range(2):
            blk = flat[n, b * 17:(b + 1) * 17]
            s = np.float32(np.array([orc.e8m0_to_f16_bits(int(blk[0]))], np.uint16).view(np.float16)[0])
            lv = np.array([s * np.float32(OCP_E2M1[c & 7] * (-1.0 if c & 8 else 1.0)) for c in range(16)], np.float32)
            for j in range(32):
                c = (blk[1 + j] & 15) if j < 16 else (blk[1 + j - 16] >> 4)
                errs = np.abs(np.float32(w[n, b * 32 + j]) - lv)
                assert c == int(np.argmax(errs == errs.min()))
    # an all-zero block gets exponent 0 and code 0 everywhere
    z = orc.quantize_rows("mxfp4", np.zeros((1, 32), np.float32))
    assert not z.any()


# ---------------------------------------------------------------------------------------------
# Q4_1: weight = d * q + m with the (d, m) pair of the row
# ---------------------------------------------------------------------------------------------
def test_q4_1_dequant_is_affine(orc):
    rng = np.random.default_rng(17)
    flat = rng.integers(0, 256, size=(8, 3 * 20), dtype=np.uint8)
    for n in range(8):                     # keep the fp16 pairs finite
        for b in range(3):
            flat[n, b * 20 + 1] &= 0x3F
            flat[n, b * 20 + 3] &= 0xBF
    deq = orc.dequantize_flat("q4_1", flat, 8, 96)
    for n in range(8):
        for b in range(3):
            blk = flat[n, b * 20:(b + 1) * 20]
            d, m = np.array([int(blk[0]) | (int(blk[1]) << 8), int(blk[2]) | (int(blk[3]) << 8)], np.uint16).view(np.float16)
            for j in range(32):
                q = (blk[4 + j] & 15) if j < 16 else (blk[4 + j - 16] >> 4)
                assert deq[n, b * 32 + j] == float(d) * q + float(m)


def test_q4_1_quantizer_hits_the_block_extremes(orc):
    w = synth.weights(16, 128, seed=23)
    flat = orc.quantize_rows("q4_1", w)
    for n in range(16):
        for b in range(4):
            blk = flat[n, b * 20:(b + 1) * 20]
            x = w[n, b * 32:(b + 1) * 32]
            d, m = np.array([int(blk[0]) | (int(blk[1]) << 8), int(blk[2]) | (int(blk[3]) << 8)], np.uint16).view(np.float16)
            assert m == np.float16(x.min())                    # m is the block minimum, rounded to fp16
            assert d == np.float16((np.float32(x.max()) - np.float32(x.min())) / np.float32(15))
            codes = [(blk[4 + j] & 15) if j < 16 else (blk[4 + j - 16] >> 4) for j in range(32)]
            assert codes[int(np.argmin(x))] == 0 and codes[int(np.argmax(x))] == 15


# ---------------------------------------------------------------------------------------------
# Q4_K ("K-Quants Formats"): super-blocks of 256, tiles = the Q4_1 tile with (d*sc, -dmin*m)
# ---------------------------------------------------------------------------------------------
def _q4k_fixture():
    spec = {"sm": [], "w": [], "pair": [], "tb": []}
    sb = np.zeros(144, np.uint8)
    for line in open(os.path.join(GOLDEN, "q4_k_superblock.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        key, vals = line[0], line[1:]
        if key == "d":
            sb[0:2] = np.array([int(vals[0], 16)], np.uint16).view(np.uint8)
        elif key == "dmin":
            sb[2:4] = np.array([int(vals[0], 16)], np.uint16).view(np.uint8)
        elif key == "scales":
            sb[4:16] = [int(v, 16) for v in vals]
        else:
            spec[key].append([int(v, 0) if key != "w" else float(v) for v in vals])
    sb[16:] = [(7 * b + 3) % 256 for b in range(128)]
    return sb, spec


def _tile_weights_q4_k(tiled, K, N):
    """Dequantize Q4_K tiles with numpy, from the tile layout alone: code = nibble of byte
    cp*32 + r, weight = fp16 d' * code + fp16 m' (the pair at 512 + 4r)."""
    nkt = K // 32
    W = np.zeros((N, K))
    for n in range(N):
        ct, r = divmod(n, 32)
        for kt in range(nkt):
            t = tiled[(ct * nkt + kt) * 640:(ct * nkt + kt + 1) * 640]
            d, m = t[512 + 4 * r:516 + 4 * r].view(np.float16).astype(np.float64)
            for c in range(32):
                b = int(t[(c // 2) * 32 + r])
                W[n, kt * 32 + c] = d * ((b >> 4) if c & 1 else (b & 15)) + m
    return W


def test_q4_k_hand_worked_superblock(orc):
    sb, spec = _q4k_fixture()
    W = orc.dequantize_flat("q4_k", sb, 1, 256)[0]
    for j, i, w in spec["w"]:
        assert W[32 * int(j) + int(i)] == w, (j, i)
    tiled = orc.repack("q4_k", sb, 256, 1)
    for kt, dbits, mbits in spec["pair"]:
        t = tiled[kt * 640:(kt + 1) * 640]
        assert int(t[512]) | (int(t[513]) << 8) == dbits and int(t[514]) | (int(t[515]) << 8) == mbits
    for kt, byte, val in spec["tb"]:
        assert tiled[kt * 640 + byte] == val
    # (sc, m) of every sub-block: with d = 1 and dmin = 0.5 the tile pair is (sc, -m/2) exactly
    for j, sc, m in spec["sm"]:
        d, mm = tiled[j * 640 + 512:j * 640 + 516].view(np.float16).astype(np.float64)
        assert d == sc and mm == -0.5 * m
    # padding rows of the tile and rows past N are zero
    assert not tiled[0 * 640 + 1:0 * 640 + 32].any()
    with pytest.raises(ValueError):
        orc.unpack("q4_k", tiled, 256, 1)


@pytest.mark.parametrize("K,N,M", [(256, 1, 1), (512, 33, 3), (768, 64, 2)])
def test_q4_k_tile_product(orc, K, N, M):
    """The tiled product equals fp64 brute force over the numpy-decoded tiles, and each tile weight is
    the flat super-block weight up to the fp16 rounding of d*sc and dmin*m (2^-11 relative each)."""
    w = synth.weights(N, K, seed=K + 3 * N)
    x = synth.activations(M, K, seed=M + 11, outliers=True)
    flat = orc.quantize_rows("q4_k", w)
    tiled = orc.repack("q4_k", flat, K, N)
    Wt = _tile_weights_q4_k(tiled, K, N)
    Wf = orc.dequantize_flat("q4_k", flat, N, K)
    mprime = np.repeat(np.abs(np.stack([tiled[(n // 32 * (K // 32) + kt) * 640 + 514 + 4 * (n % 32):][:2].view(np.float16)[0]
                                        for n in range(N) for kt in range(K // 32)]).astype(np.float64).reshape(N, K // 32)), 32, axis=1)
    assert np.all(np.abs(Wt - Wf) <= 2.0 ** -11 * (np.abs(Wf) + 2.001 * mprime) + 1e-30)
    a_q, a_d = orc.quantize_act(x)
    y, bound = orc.matmul("q4_k", tiled, K, N, a_q, a_d)
    A = a_q.astype(np.float64) * np.repeat(a_d.view(np.float16).astype(np.float64), 32, axis=1)
    assert np.allclose(y, A @ Wt.T, rtol=1e-12, atol=1e-15)
    assert np.allclose(bound, np.abs(A) @ np.abs(Wt).T, rtol=1e-12, atol=1e-15)
    y41, _ = orc.matmul("q4_1", tiled, K, N, a_q, a_d)     # the same tile read as Q4_1
    assert np.array_equal(y, y41)


def test_q4_k_quantizer_error_bound(orc):
    """|x - dequant| <= max(D/2, 15 |scale - D| + |min - M|) per sub-block, with the scale and min
    errors bounded by the 6-bit rounding against d = max scale / 63 and dmin = max min / 63."""
    K, N = 512, 24
    w = synth.weights(N, K, seed=31)
    w[3, :256] = 0.0                                  # an all-zero super-block
    w[5, 256:] = np.abs(w[5, 256:])                   # a super-block with no negative element
    flat = orc.quantize_rows("q4_k", w)
    Wf = orc.dequantize_flat("q4_k", flat, N, K)
    for n in range(N):
        for s in range(K // 256):
            x = w[n, 256 * s:256 * (s + 1)].astype(np.float64).reshape(8, 32)
            mn = np.minimum(0.0, x.min(axis=1))
            scale = (x.max(axis=1) - mn) / 15
            d, dmin = scale.max() / 63, (-mn).max() / 63
            e_scale = (0.5 + 63 * 2.0 ** -11) * d + 1e-12
            e_min = (0.5 + 63 * 2.0 ** -11) * dmin + 1e-12
            err = np.abs(x - Wf[n, 256 * s:256 * (s + 1)].reshape(8, 32)).max(axis=1)
            lim = np.maximum((scale + e_scale) / 2, 15 * e_scale + e_min) * (1 + 1e-5) + 1e-9
            assert np.all(err <= lim), (n, s, err, lim)
    assert not Wf[3, :256].any()


def test_activation_arrays_are_ggml_q8_0_blocks(orc):
    """a_q / a_d hold the same values as GGML Q8_0 blocks: packed as {d, qs[32]} they equal, byte for
    byte, the Q8_0 quantization of the same rows through the flat-block writer (a separate code path
    that applies the same rule), and unpack back unchanged."""
    x = synth.activations(5, 256, seed=77, outliers=True)
    x[1, :32] = 0.0
    a_q, a_d = orc.quantize_act(x)
    blocks = orc.act_to_blocks(a_q, a_d)
    assert np.array_equal(blocks, orc.quantize_rows("q8_0", x))
    q2, d2 = orc.blocks_to_act(blocks, 5, 256)
    assert np.array_equal(q2, a_q) and np.array_equal(d2, a_d)


def test_q4_k_quantizer_hand_case(orc):
    """Sub-block 0 spans [0, 15] (scale 1), sub-block 1 spans [0, 7.5] (scale 0.5), the rest are zero,
    nothing is negative.  By hand: d = fp16(1/63) = 0x2410, dmin = 0; sc_0 = trunc(1*63 + 0.5) = 63,
    sc_1 = trunc(0.5*63 + 0.5) = 32 (31 if the 6-bit scales were truncated instead of rounded);
    f32(d) = 1.015625/64, so 15 and 7.5 both land on code 15 and the zeros on code 0."""
    x = np.zeros((1, 256), np.float32)
    x[0, 1] = 15.0
    x[0, 33] = 7.5
    sb = orc.quantize_rows("q4_k", x)[0]
    assert int(sb[0]) | (int(sb[1]) << 8) == 0x2410
    assert int(sb[2]) | (int(sb[3]) << 8) == 0
    assert sb[4] & 63 == 63 and sb[5] & 63 == 32
    assert not (sb[6:8] & 63).any() and not (sb[8:12] & 63).any()
    codes = [(sb[16 + 32 * (j // 2) + i] >> (4 * (j & 1))) & 15 for j in range(2) for i in range(32)]
    assert codes[1] == 15 and codes[33] == 15
    assert sum(codes) == 30

"""GPU parity for Q4_K ("K-Quants Formats"): GGML super-blocks of 256 weights, repacked into the Q4_1
tile with the row pair (fp16(d*sc), fp16(-dmin*m)).

Bit-exact for the byte work (the weight quantizer and the repack); every matmul path (decode,
tensor-core GEMM, fused activation quantization, flat rows) within
|gpu - oracle| <= 1e-5 * sum_k |w_k * x_k| + 1e-6 of the oracle's fp64 product over its own tiles.
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import (assert_within_bound, dev_u8, gpu_matmul, gpu_matmul_f32, gpu_matmul_ws,
                            gpu_prepare_weight, gpu_quantize_act, torch_mod)

pytestmark = pytest.mark.gpu
T = "q4_k"


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _special_rows(K):
    rows = [np.zeros(K, np.float32)]                                   # all-zero super-blocks
    r = np.abs(synth.weights(1, K, seed=1)[0]); rows.append(r)         # no negative element (min 0)
    r = -np.abs(synth.weights(1, K, seed=2)[0]); rows.append(r)        # no positive element
    r = np.zeros(K, np.float32); r[::32] = 1.0; rows.append(r)         # one non-zero per sub-block
    r = np.full(K, 1e-30, np.float32); rows.append(r)                  # tiny scales (fp16 underflow)
    r = synth.weights(1, K, seed=3)[0] * 5e7; rows.append(r)           # d*sc beyond fp16 range
    r = np.linspace(-1, 1, K, dtype=np.float32); r[:32] = -0.0; rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("N,K", [(1, 256), (33, 512), (100, 1024), (7, 512)])
def test_q4_k_quantize_and_repack_bit_exact(torch, orc, N, K):
    w = _special_rows(K) if N == 7 else synth.weights(N, K, seed=N * 7 + K)
    flat_d, tiled_d = gpu_prepare_weight(T, w)
    flat_ref = orc.quantize_rows(T, w)
    assert np.array_equal(flat_d.cpu().numpy(), flat_ref.reshape(-1)), "quantize_weight"
    assert np.array_equal(tiled_d.cpu().numpy(), orc.repack(T, flat_ref, K, N)), "repack"


@pytest.mark.parametrize("N,K", [(1, 256), (33, 512), (4096 + 5, 256)])
def test_q4_k_repack_random_superblocks(torch, orc, N, K):
    import block_quantized_matmul_gb300 as qmm

    rng = np.random.default_rng(N + K)
    flat = rng.integers(0, 256, size=(N, K // 256, 144), dtype=np.uint8)
    flat[:, :, 1] &= 0x3F                    # d and dmin finite (exponent below 0x1F)
    flat[:, :, 3] &= 0xBF
    flat = flat.reshape(N, -1)
    tiled_d = torch.full((qmm.tiled_size(T, K, N),), 0x5A, dtype=torch.uint8, device="cuda")
    qmm.qmm_repack(T, dev_u8(flat), K, N, tiled_d)
    assert np.array_equal(tiled_d.cpu().numpy(), orc.repack(T, flat, K, N))


def _case(torch, orc, N, K, M, path, ldy=None, outliers=False):
    w = synth.weights(N, K, seed=3 * N + K)
    x = synth.activations(M, K, seed=M * 11 + K, outliers=outliers)
    flat_ref = orc.quantize_rows(T, w)
    tiled_ref = orc.repack(T, flat_ref, K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(T, tiled_ref, K, N, q_ref, d_ref)
    flat_d, tiled_d = gpu_prepare_weight(T, w)
    a_q, a_d = gpu_quantize_act(x)
    ys = {}
    if path in ("decode", "gemm"):
        ys[path] = gpu_matmul(T, tiled_d, K, N, a_q, a_d, M, path=1 if path == "decode" else 2, ldy=ldy)
    if path == "ws":
        ys[path] = gpu_matmul_ws(T, tiled_d, K, N, a_q, a_d, M, ldy=ldy)
    if path == "fused":
        ys[path] = gpu_matmul_f32(T, tiled_d, K, N, x, ldy=ldy)
    if path == "flat":
        import block_quantized_matmul_gb300 as qmm

        y = torch.full((M, ldy or N), float("nan"), dtype=torch.float32, device="cuda")
        qmm.qmm_matmul_flat(T, flat_d, K, N, a_q, a_d, M, y, ldy or N)
        torch.cuda.synchronize()
        ys[path] = y
    for name, y in ys.items():
        yh = y.cpu().numpy()
        assert_within_bound(yh[:, :N], y_ref, bound, f"{name} q4_k N={N} K={K} M={M}")
        if ldy is not None and ldy > N:
            assert np.isnan(yh[:, N:]).all()


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("N,K", [(100, 256), (33, 1024), (300, 4096)])
@pytest.mark.parametrize("path", ["decode", "fused", "flat"])
def test_q4_k_decode_paths(torch, orc, path, M, N, K):
    _case(torch, orc, N, K, M, path)


@pytest.mark.parametrize("M", [1, 17, 128, 300])
@pytest.mark.parametrize("N,K", [(100, 256), (544, 1024)])
@pytest.mark.parametrize("path", ["gemm", "ws"])
def test_q4_k_gemm_paths(torch, orc, path, M, N, K):
    _case(torch, orc, N, K, M, path, outliers=True)


def test_q4_k_ragged_ldy_and_k_passes(torch, orc):
    _case(torch, orc, 31, 256, 3, "decode", ldy=40)
    _case(torch, orc, 31, 256, 3, "flat", ldy=40)
    _case(torch, orc, 70, 256 * 50, 2, "decode")      # K passes of the staged activations
    _case(torch, orc, 70, 256 * 50, 2, "flat")
    _case(torch, orc, 65, 512, 129, "gemm", ldy=70)


@pytest.mark.parametrize("M", [1, 512])
def test_q4_k_full_size_sampled(torch, orc, M):
    K, N = 4096, 14336
    w = synth.weights(N, K)
    x = synth.activations(M, K)
    flat_ref = orc.quantize_rows(T, w)
    tiled_ref = orc.repack(T, flat_ref, K, N)
    del flat_ref
    q_ref, d_ref = orc.quantize_act(x)
    _, tiled_d = gpu_prepare_weight(T, w)
    del w
    step = 1 << 26
    for s in range(0, tiled_ref.size, step):
        assert np.array_equal(tiled_d[s:s + step].cpu().numpy(), tiled_ref[s:s + step]), f"tiles @ {s}"
    if M == 1:
        y = gpu_matmul_f32(T, tiled_d, K, N, x).cpu().numpy()
    else:
        a_q, a_d = gpu_quantize_act(x)
        y = gpu_matmul_ws(T, tiled_d, K, N, a_q, a_d, M).cpu().numpy()
    rng = np.random.default_rng(0)
    n_ct = (N + 31) // 32
    ns = np.concatenate([np.arange(n_ct) * 32 + rng.integers(0, 32, n_ct), [0, N - 1]]).clip(0, N - 1)
    ms = rng.integers(0, M, ns.size)
    ys, bs = orc.matmul_at(T, tiled_ref, K, q_ref, d_ref, ms, ns)
    assert_within_bound(y[ms, ns], ys, bs, f"q4_k {K}x{N} M={M}")
    assert np.isfinite(y).all()

"""GPU parity of qmm_matmul_flat, the decode matmul taken straight from flat GGML rows.

The flat bytes fed to the GPU are the oracle's own quantized rows; the expected values are the
oracle's fp64 product and bound over the same blocks, and the GPU result must lie within
|gpu - oracle| <= 1e-5 * sum_k |w_k * x_k| + 1e-6 per element.
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import TYPES, assert_within_bound, dev_u8, gpu_quantize_act, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _flat_matmul(torch, type_, flat_d, K, N, a_q, a_d, M, ldy=None):
    import block_quantized_matmul_gb300 as qmm

    ldy = N if ldy is None else ldy
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_matmul_flat(type_, flat_d, K, N, a_q, a_d, M, y, ldy)
    torch.cuda.synchronize()
    return y


def _case(torch, orc, type_, N, K, M, ldy=None, outliers=False):
    w = synth.weights(N, K, seed=17 * N + K)
    x = synth.activations(M, K, seed=M * 19 + K, outliers=outliers)
    flat_ref = orc.quantize_rows(type_, w)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, orc.repack(type_, flat_ref, K, N), K, N, q_ref, d_ref)
    a_q, a_d = gpu_quantize_act(x)
    y = _flat_matmul(torch, type_, dev_u8(flat_ref), K, N, a_q, a_d, M, ldy=ldy).cpu().numpy()
    assert_within_bound(y[:, :N], y_ref, bound, f"flat {type_} N={N} K={K} M={M}")
    if ldy is not None and ldy > N:
        assert np.isnan(y[:, N:]).all(), "columns past N must stay untouched"


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9])
@pytest.mark.parametrize("N,K", [(100, 512), (33, 1024), (300, 4096)])
def test_flat_parity(torch, orc, type_, M, N, K):
    _case(torch, orc, type_, N, K, M)


@pytest.mark.parametrize("type_", TYPES)
def test_flat_ragged_ldy_and_k_passes(torch, orc, type_):
    _case(torch, orc, type_, 1, 512, 1)                       # one row
    _case(torch, orc, type_, 31, 512, 3, ldy=40, outliers=True)
    _case(torch, orc, type_, 70, 32 * 400, 2)                 # two passes over K, the last stage half full
    _case(torch, orc, type_, 45, 32 * 800, 4)                 # three passes


def test_flat_other_row_lengths(torch, orc):
    """Row lengths that are 16-byte multiples without K % 512 == 0."""
    _case(torch, orc, "q4_0", 50, 32 * 8, 1)                  # 8 blocks of 18 B
    _case(torch, orc, "q4_1", 50, 32 * 4, 2)                  # 4 blocks of 20 B
    _case(torch, orc, "q8_0", 50, 32 * 24, 3)                 # 24 blocks of 34 B


def test_flat_matches_tiled_decode(torch, orc):
    """The flat and tiled decode paths agree within the bound on the same blocks."""
    from tests.gpu_util import gpu_matmul, gpu_prepare_weight

    K, N, M = 2048, 640, 4
    w = synth.weights(N, K, seed=3)
    x = synth.activations(M, K, seed=4)
    for type_ in TYPES:
        flat_d, tiled_d = gpu_prepare_weight(type_, w)
        a_q, a_d = gpu_quantize_act(x)
        y_flat = _flat_matmul(torch, type_, flat_d, K, N, a_q, a_d, M).cpu().numpy()
        y_tiled = gpu_matmul(type_, tiled_d, K, N, a_q, a_d, M, path=1).cpu().numpy()
        q_ref, d_ref = orc.quantize_act(x)
        _, bound = orc.matmul(type_, orc.repack(type_, orc.quantize_rows(type_, w), K, N), K, N, q_ref, d_ref)
        assert_within_bound(y_flat, y_tiled.astype(np.float64), 2 * bound, f"flat vs tiled {type_}")


FULL = [("q4_0", 4096, 14336, 1), ("q8_0", 4096, 4096, 1), ("mxfp4", 4096, 14336, 1), ("iq4_nl", 14336, 4096, 4)]


@pytest.mark.parametrize("type_,K,N,M", FULL, ids=lambda v: str(v))
def test_flat_full_size_sampled(torch, orc, type_, K, N, M):
    w = synth.weights(N, K)
    x = synth.activations(M, K)
    flat_ref = orc.quantize_rows(type_, w)
    del w
    q_ref, d_ref = orc.quantize_act(x)
    a_q, a_d = gpu_quantize_act(x)
    y = _flat_matmul(torch, type_, dev_u8(flat_ref), K, N, a_q, a_d, M).cpu().numpy()
    tiled_ref = orc.repack(type_, flat_ref, K, N)
    rng = np.random.default_rng(1)
    n_ct = (N + 31) // 32
    ns = np.concatenate([np.arange(n_ct) * 32 + rng.integers(0, 32, n_ct), [0, N - 1]]).clip(0, N - 1)
    ms = rng.integers(0, M, ns.size)
    ys, bs = orc.matmul_at(type_, tiled_ref, K, q_ref, d_ref, ms, ns)
    assert_within_bound(y[ms, ns], ys, bs, f"flat {type_} {K}x{N} M={M}")
    assert np.isfinite(y).all()

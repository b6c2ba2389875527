"""GPU parity of the exact-integer tensor-core GEMM at long K, against the CPU oracle.

The GEMM sums each output's blocks in an fp32 register for at most 128 blocks (K = 4096) and then
adds that chunk into y, so its error bound is (128 + K/4096) * 2^-24 * sum_k |w_k x_k|, inside
the 1e-5 tolerance up to the largest accepted K (131072).  These cases run it where one
accumulator over all of K would not be inside the bound in the worst case: an FFN down-projection
shape (K = 14336, several chunks and a partial last one), all-positive operands (every rounding
pushes the same way), and K = 32768 checked element by element.  Bound: |gpu - oracle| <=
1e-5 * sum_k |w_k x_k| + 1e-6 per element.
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import assert_within_bound, gpu_matmul, gpu_matmul_ws, gpu_prepare_weight, gpu_quantize_act, torch_mod

pytestmark = pytest.mark.gpu
AUTO, GEMM = 0, 2


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _columns(N):
    """One column per column tile (a different row of each tile) plus both ends."""
    rng = np.random.default_rng(N)
    n_ct = (N + 31) // 32
    return np.unique(np.concatenate([np.arange(n_ct) * 32 + rng.integers(0, 32, n_ct), [0, N - 1]]).clip(0, N - 1))


def _inputs(type_, N, K, M, positive, seed):
    w = synth.weights(N, K, seed=seed)
    x = synth.activations(M, K, seed=seed + 1, outliers=not positive)
    if positive:
        w, x = np.abs(w), np.abs(x)
    return w, x


@pytest.mark.parametrize("type_", ["q4_0", "q8_0"])
@pytest.mark.parametrize("positive", [False, True], ids=["signed", "all_positive"])
def test_ffn_down_projection_shape(torch, orc, type_, positive):
    import block_quantized_matmul_gb300 as qmm

    K, N, M = 14336, 4096, 512
    w, x = _inputs(type_, N, K, M, positive, seed=61)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    _, tiled = gpu_prepare_weight(type_, w)
    a_q, a_d = gpu_quantize_act(x)
    assert np.array_equal(a_q.cpu().numpy(), q_ref)
    cols = _columns(N)
    ms = np.repeat(np.arange(M), cols.size)
    ns = np.tile(cols, M)
    ys, bs = orc.matmul_at(type_, tiled_ref, K, q_ref, d_ref, ms, ns)
    for what, y in (("gemm", gpu_matmul(type_, tiled, K, N, a_q, a_d, M, path=GEMM)),
                    ("auto", gpu_matmul(type_, tiled, K, N, a_q, a_d, M, path=AUTO)),
                    ("workspace", gpu_matmul_ws(type_, tiled, K, N, a_q, a_d, M))):
        assert qmm.qmm_device_status() == 0
        y = y.cpu().numpy()
        assert np.isfinite(y).all()
        assert_within_bound(y[ms, ns], ys, bs, f"{what} {type_} K={K} positive={positive}")


@pytest.mark.parametrize("type_", ["q4_0", "iq4_nl", "q4_1"])
def test_k32768_elementwise(torch, orc, type_):
    import block_quantized_matmul_gb300 as qmm

    K, N, M = 32768, 160, 136
    w, x = _inputs(type_, N, K, M, positive=True, seed=62)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
    _, tiled = gpu_prepare_weight(type_, w)
    a_q, a_d = gpu_quantize_act(x)
    y = gpu_matmul(type_, tiled, K, N, a_q, a_d, M, path=GEMM).cpu().numpy()
    assert qmm.qmm_device_status() == 0
    assert_within_bound(y, y_ref, bound, f"gemm {type_} K={K}")

"""GPU parity of the tensor-core (tcgen05) GEMM path against the CPU oracle.

|gpu - oracle| <= 1e-5 * sum_k |w_k * x_k| + 1e-6 per element; shapes span several 128 x 128
output tiles with ragged token counts (M) and ragged weight-row counts (N, including N with a
column-tile count that is not a multiple of 4).
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import (TYPES, assert_within_bound, gpu_matmul, gpu_matmul_ws, gpu_prepare_weight, oracle_at_parallel,
                            gpu_quantize_act, torch_mod)

pytestmark = pytest.mark.gpu
GEMM = 2


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _case(torch, orc, type_, N, K, M, outliers=True, ldy=None, ws=False):
    import block_quantized_matmul_gb300 as qmm

    w = synth.weights(N, K, seed=5 * N + K)
    x = synth.activations(M, K, seed=M * 13 + K, outliers=outliers)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
    _, tiled_d = gpu_prepare_weight(type_, w)
    a_q, a_d = gpu_quantize_act(x)
    if ws:
        y = gpu_matmul_ws(type_, tiled_d, K, N, a_q, a_d, M, ldy=ldy).cpu().numpy()
    else:
        y = gpu_matmul(type_, tiled_d, K, N, a_q, a_d, M, path=GEMM, ldy=ldy).cpu().numpy()
    assert qmm.qmm_device_status() == 0
    assert_within_bound(y[:, :N], y_ref, bound, f"gemm {type_} N={N} K={K} M={M} ws={ws}")
    if ldy is not None and ldy > N:
        assert np.isnan(y[:, N:]).all()
    return y


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 17, 128, 129, 300])
@pytest.mark.parametrize("N,K", [(128, 64), (100, 256), (544, 1024)])
def test_gemm_parity(torch, orc, type_, M, N, K):
    _case(torch, orc, type_, N, K, M)


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [17, 128, 129, 300])
@pytest.mark.parametrize("N,K", [(100, 256), (544, 1024)])
def test_gemm_workspace_parity(torch, orc, type_, M, N, K):
    _case(torch, orc, type_, N, K, M, ws=True)


@pytest.mark.parametrize("type_", TYPES)
def test_gemm_workspace_ragged(torch, orc, type_):
    _case(torch, orc, type_, 33, 32, 19, ws=True)              # one K tile, M not a multiple of 8
    _case(torch, orc, type_, 31, 96, 130, ldy=48, ws=True)
    _case(torch, orc, type_, 4100, 128, 40, ws=True)


@pytest.mark.parametrize("type_", ["mxfp4", "q4_1"])
def test_gemm_workspace_matches_in_kernel_path(torch, type_):
    # tile types without a folded-scale kernel: the workspace path is the exact-integer kernel with a
    # prepared token operand -> same integers and scales as the in-kernel variant, identical results
    w = synth.weights(512, 1024, seed=21)
    x = synth.activations(200, 1024, seed=22, outliers=True)
    _, tiled = gpu_prepare_weight(type_, w)
    a_q, a_d = gpu_quantize_act(x)
    y1 = gpu_matmul(type_, tiled, 1024, 512, a_q, a_d, 200, path=GEMM)
    y2 = gpu_matmul_ws(type_, tiled, 1024, 512, a_q, a_d, 200)
    y3 = gpu_matmul_ws(type_, tiled, 1024, 512, a_q, a_d, 200, fill=0xFF)
    assert torch.equal(y1, y2) and torch.equal(y2, y3)


def test_gemm_workspace_contents_do_not_matter(torch):
    # the folded-scale kernel writes every workspace byte it reads: a dirty workspace changes nothing
    w = synth.weights(512, 1024, seed=21)
    x = synth.activations(200, 1024, seed=22, outliers=True)
    _, tiled = gpu_prepare_weight("q4_0", w)
    a_q, a_d = gpu_quantize_act(x)
    y2 = gpu_matmul_ws("q4_0", tiled, 1024, 512, a_q, a_d, 200)
    y3 = gpu_matmul_ws("q4_0", tiled, 1024, 512, a_q, a_d, 200, fill=0xFF)
    assert torch.equal(y2, y3)


@pytest.mark.parametrize("type_", TYPES)
def test_gemm_ragged_and_ldy(torch, orc, type_):
    _case(torch, orc, type_, 33, 32, 5)               # one K tile, one partial column tile
    _case(torch, orc, type_, 31, 96, 130, ldy=48)     # ldy > N, token tail
    _case(torch, orc, type_, 4100, 128, 40)           # 129 column tiles: last CTA holds 1 of 4


def test_gemm_matches_matvec(torch, orc):
    # the two kernels implement the same formula: both within the bound, and close to each other
    w = synth.weights(256, 2048, seed=3)
    x = synth.activations(16, 2048, seed=4, outliers=True)
    _, tiled = gpu_prepare_weight("q4_0", w)
    a_q, a_d = gpu_quantize_act(x)
    y_mv = gpu_matmul("q4_0", tiled, 2048, 256, a_q, a_d, 16, path=1).cpu().numpy()
    y_tc = gpu_matmul("q4_0", tiled, 2048, 256, a_q, a_d, 16, path=GEMM).cpu().numpy()
    assert np.allclose(y_mv, y_tc, rtol=1e-4, atol=1e-4)


def test_gemm_is_deterministic(torch):
    w = synth.weights(512, 1024, seed=8)
    x = synth.activations(256, 1024, seed=9)
    _, tiled = gpu_prepare_weight("q8_0", w)
    a_q, a_d = gpu_quantize_act(x)
    y1 = gpu_matmul("q8_0", tiled, 1024, 512, a_q, a_d, 256, path=GEMM)
    y2 = gpu_matmul("q8_0", tiled, 1024, 512, a_q, a_d, 256, path=GEMM)
    assert torch.equal(y1, y2)


FULL = [("q4_0", 4096, 14336, 512), ("q8_0", 4096, 128256, 128), ("mxfp4", 4096, 14336, 512),
        ("q4_1", 4096, 14336, 512)]
# the prefill and batched lm-head workloads: checked on a dense grid (all rows x ~1024 or 4010 columns)
DENSE = {("q4_0", 4096, 14336, 512), ("q8_0", 4096, 128256, 128)}


@pytest.mark.parametrize("type_,K,N,M", FULL, ids=lambda v: str(v))
def test_gemm_full_size_sampled(torch, orc, type_, K, N, M):
    import block_quantized_matmul_gb300 as qmm

    w = synth.weights(N, K)
    x = synth.activations(M, K, outliers=(type_ == "q4_0"))
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    _, tiled_d = gpu_prepare_weight(type_, w)
    del w
    step = 1 << 26
    for s in range(0, tiled_ref.size, step):
        assert np.array_equal(tiled_d[s:s + step].cpu().numpy(), tiled_ref[s:s + step]), f"tiles @ {s}"
    a_q, a_d = gpu_quantize_act(x)
    y = gpu_matmul(type_, tiled_d, K, N, a_q, a_d, M, path=0).cpu().numpy()
    y_ws = gpu_matmul_ws(type_, tiled_d, K, N, a_q, a_d, M).cpu().numpy()
    if type_ in ("mxfp4", "q4_1"):         # same exact-integer kernel either way
        assert np.array_equal(y, y_ws)
    assert qmm.qmm_device_status() == 0
    rng = np.random.default_rng(1)
    n_ct = (N + 31) // 32
    if (type_, K, N, M) in DENSE:
        # every token row x (one column in every column tile, random columns up to 1024 where there
        # are fewer tiles, and both ends); the oracle runs on a spawned process pool
        cols = np.arange(n_ct) * 32 + rng.integers(0, 32, n_ct)
        cols = np.concatenate([cols, rng.integers(0, N, max(0, 1024 - n_ct - 2)), [0, N - 1]])
        cols = np.unique(cols.clip(0, N - 1))
        ms, ns = np.repeat(np.arange(M), cols.size), np.tile(cols, M)
        ys, bs = oracle_at_parallel(type_, tiled_ref, K, q_ref, d_ref, ms, ns)
    else:
        ns = np.concatenate([np.arange(n_ct) * 32 + rng.integers(0, 32, n_ct), [0, N - 1, N - 1]]).clip(0, N - 1)
        ms = np.concatenate([rng.integers(0, M, n_ct), [0, M - 1, 0]])
        ys, bs = orc.matmul_at(type_, tiled_ref, K, q_ref, d_ref, ms, ns)
    assert_within_bound(y[ms, ns], ys, bs, f"gemm {type_} {K}x{N} M={M}")
    assert_within_bound(y_ws[ms, ns], ys, bs, f"gemm (workspace) {type_} {K}x{N} M={M}")
    assert np.isfinite(y).all() and np.isfinite(y_ws).all()

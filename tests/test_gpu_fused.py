"""GPU parity of qmm_matmul_f32, the decode matmul with the activation quantization fused in.

Against the oracle (quantize the fp32 rows, then the fp64 product and bound) within
|gpu - oracle| <= 1e-5 * sum_k |w_k * x_k| + 1e-6, and bit for bit against the two-call path
(qmm_quantize_act + the decode matmul), which applies the same quantization rule and the same
accumulation order.
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import (TYPES, assert_within_bound, gpu_matmul, gpu_matmul_f32, gpu_prepare_weight,
                            gpu_quantize_act, torch_mod)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _case(torch, orc, type_, N, K, M, ldx=None, ldy=None, x_offset=0, outliers=False):
    w = synth.weights(N, K, seed=7 * N + K)
    x = synth.activations(M, K, seed=M * 13 + K, outliers=outliers)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
    _, tiled = gpu_prepare_weight(type_, w)
    y = gpu_matmul_f32(type_, tiled, K, N, x, ldx=ldx, ldy=ldy, x_offset=x_offset)
    yh = y.cpu().numpy()
    assert_within_bound(yh[:, :N], y_ref, bound, f"fused {type_} N={N} K={K} M={M}")
    if ldy is not None and ldy > N:
        assert np.isnan(yh[:, N:]).all(), "columns past N must stay untouched"
    # the two-call path gives the same bits
    a_q, a_d = gpu_quantize_act(x)
    y2 = gpu_matmul(type_, tiled, K, N, a_q, a_d, M, path=1, ldy=ldy)
    assert torch.equal(y[:, :N], y2[:, :N])


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16, 17])
@pytest.mark.parametrize("N,K", [(100, 256), (33, 1056), (300, 4096)])
def test_fused_parity(torch, orc, type_, M, N, K):
    _case(torch, orc, type_, N, K, M)


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 3, 12])
def test_fused_strided_and_unaligned_rows(torch, orc, type_, M):
    _case(torch, orc, type_, 65, 320, M, ldx=333, ldy=70)        # ldx odd: scalar loads
    _case(torch, orc, type_, 65, 320, M, ldx=324, x_offset=1)    # rows 4-byte aligned only
    _case(torch, orc, type_, 31, 32, M, ldx=36, outliers=True)   # one tile of K


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 4, 16])
def test_fused_k_passes(torch, orc, type_, M):
    _case(torch, orc, type_, 70, 32 * 1100, M)


def test_fused_special_blocks(torch, orc):
    """All-zero blocks, a lone maximum, exact .5 ties and tiny magnitudes go through the fused
    quantizer exactly as through qmm_quantize_act."""
    K = 256
    x = np.zeros((4, K), np.float32)
    x[1, 0] = 3.0
    x[1, 1:32] = np.linspace(-1.0, 1.0, 31, dtype=np.float32)
    x[2, :] = np.tile(np.array([127.0, 2.5, -2.5, 0.5, -0.5, 1.5], np.float32), K // 6 + 1)[:K]
    x[3, :] = np.float32(1e-30)
    x[3, ::5] = np.float32(-3e-39)
    _case_x(torch, orc, "q8_0", 40, K, x)
    _case_x(torch, orc, "q4_0", 40, K, x)


def _case_x(torch, orc, type_, N, K, x):
    w = synth.weights(N, K, seed=5)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
    _, tiled = gpu_prepare_weight(type_, w)
    y = gpu_matmul_f32(type_, tiled, K, N, x)
    assert_within_bound(y.cpu().numpy(), y_ref, bound, f"fused specials {type_}")
    a_q, a_d = gpu_quantize_act(x)
    assert torch.equal(y, gpu_matmul(type_, tiled, K, N, a_q, a_d, x.shape[0], path=1))


FULL = [("q4_0", 4096, 4096, 1), ("q8_0", 4096, 14336, 1), ("iq4_nl", 4096, 4096, 8), ("q8_0", 4096, 128256, 1)]


@pytest.mark.parametrize("type_,K,N,M", FULL, ids=lambda v: str(v))
def test_fused_full_size_sampled(torch, orc, type_, K, N, M):
    w = synth.weights(N, K)
    x = synth.activations(M, K)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    _, tiled = gpu_prepare_weight(type_, w)
    del w
    y = gpu_matmul_f32(type_, tiled, K, N, x).cpu().numpy()
    rng = np.random.default_rng(1)
    n_ct = (N + 31) // 32
    ns = np.concatenate([np.arange(n_ct) * 32 + rng.integers(0, 32, n_ct), [0, N - 1]]).clip(0, N - 1)
    ms = rng.integers(0, M, ns.size)
    ys, bs = orc.matmul_at(type_, tiled_ref, K, q_ref, d_ref, ms, ns)
    assert_within_bound(y[ms, ns], ys, bs, f"fused {type_} {K}x{N} M={M}")
    assert np.isfinite(y).all()


@pytest.mark.parametrize("type_", ["q8_0", "q4_0"])
@pytest.mark.parametrize("M", [1, 4, 9])
def test_fused_with_host_buffers(torch, orc, type_, M):
    """x and y in page-locked host memory, handed to the call as they are: the kernel reads and
    writes them over the host link; the result equals the device-buffer call bit for bit."""
    import block_quantized_matmul_gb300 as qmm

    K, N = 1024, 300
    w = synth.weights(N, K, seed=41)
    x = synth.activations(M, K, seed=42)
    _, tiled = gpu_prepare_weight(type_, w)
    y_dev = gpu_matmul_f32(type_, tiled, K, N, x)
    x_host = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    y_host = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    qmm.qmm_matmul_f32(type_, tiled, K, N, x_host, K, M, y_host, N)
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu())
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, orc.repack(type_, orc.quantize_rows(type_, w), K, N), K, N, q_ref, d_ref)
    assert_within_bound(y_host.numpy(), y_ref, bound, f"host buffers {type_} M={M}")

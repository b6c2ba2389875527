"""GPU parity of the folded-scale tensor-core GEMM against the CPU oracle.

qmm_matmul_ws (and qmm_matmul_noalloc) run Q4_0, Q8_0 and IQ4_NL prefill shapes on the kernel that
folds the block scales into exact hi + lo fp16 operands and accumulates 128-wide K chunks in fp32 on
the tensor cores (K in passes of at most 4096 added into y).  Bound: |gpu - oracle| <= 1e-5 * sum_k |w_k x_k| + 1e-6 per element.  Beyond the
shapes of test_gpu_gemm.py these cases aim at what is particular to that kernel:
  * long K with a partial last chunk and an odd number of blocks (K = 4192: 131 blocks);
  * all-positive operands, where every rounding of the fp32 accumulation pushes the same way;
  * token rows and weight rows large enough to take the power-of-two range shift, including rows
    whose blocks differ in magnitude by 10^6, and rows whose small block scales cannot survive the
    shift (the call reports QMM_ERR_RANGE; the exact-integer path computes them);
  * operands at the other end of fp16's range (tiny block scales, subnormal lo terms).
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import assert_within_bound, gpu_matmul_ws, gpu_prepare_weight, gpu_quantize_act, torch_mod

pytestmark = pytest.mark.gpu
FOLD_TYPES = ["q4_0", "q8_0", "iq4_nl"]


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _run(orc, type_, w, x, what, ldy=None):
    import block_quantized_matmul_gb300 as qmm

    N, K = w.shape
    M = x.shape[0]
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
    _, tiled_d = gpu_prepare_weight(type_, w)
    a_q, a_d = gpu_quantize_act(x)
    assert np.array_equal(tiled_d.cpu().numpy(), tiled_ref)
    assert np.array_equal(a_q.cpu().numpy(), q_ref)
    y = gpu_matmul_ws(type_, tiled_d, K, N, a_q, a_d, M, ldy=ldy).cpu().numpy()
    assert qmm.qmm_device_status() == 0
    assert_within_bound(y[:, :N], y_ref, bound, f"fold {type_} {what} N={N} K={K} M={M}")
    return y


@pytest.mark.parametrize("type_", FOLD_TYPES)
@pytest.mark.parametrize("N,K,M", [(256, 4192, 150), (96, 8192, 40), (4100, 64, 257)])
def test_fold_shapes(torch, orc, type_, N, K, M):
    w = synth.weights(N, K, seed=N + K)
    x = synth.activations(M, K, seed=M + K, outliers=True)
    _run(orc, type_, w, x, "shape")


@pytest.mark.parametrize("type_", FOLD_TYPES)
def test_fold_all_positive(torch, orc, type_):
    w = np.abs(synth.weights(160, 4096, seed=41))
    x = np.abs(synth.activations(130, 4096, seed=42))
    _run(orc, type_, w, x, "all positive")


@pytest.mark.parametrize("type_", FOLD_TYPES)
def test_fold_token_range_shift(torch, orc, type_):
    x = synth.activations(140, 1024, seed=43, outliers=True)
    # (block maxima stay below 127 * 65504, where the Q8_0 rule's fp16 scale itself would overflow)
    x[3] *= np.float32(5e4)                 # 127 * d_a far beyond 2^15: shifted row
    x[77, :512] *= np.float32(2e4)          # half a row large, half ordinary: one shift for both
    x[90] *= np.float32(1e-6)               # tiny scales (subnormal lo terms), no shift
    w = synth.weights(200, 1024, seed=44)
    _run(orc, type_, w, x, "token range")


@pytest.mark.parametrize("type_", FOLD_TYPES)
def test_fold_weight_range_shift(torch, orc, type_):
    w = synth.weights(200, 1024, seed=45)
    w[5] *= np.float32(1e6)                 # |d_w| * max|w_int| beyond 2^15: shifted row
    w[40, :256] *= np.float32(1e6)          # one row with large and ordinary blocks
    w[130] *= np.float32(1e-3)              # tiny block scales
    x = synth.activations(150, 1024, seed=46)
    _run(orc, type_, w, x, "weight range")


RANGE = 6          # QMM_ERR_RANGE


def _range_case(torch, orc, type_, w, x, what):
    """The folded-scale path reports the call (its result is then not exact); the exact-integer path
    computes the same data within the bound."""
    import block_quantized_matmul_gb300 as qmm
    from tests.gpu_util import gpu_matmul

    N, K = w.shape
    M = x.shape[0]
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
    _, tiled = gpu_prepare_weight(type_, w)
    a_q, a_d = gpu_quantize_act(x)
    assert qmm.qmm_device_status() == 0
    gpu_matmul_ws(type_, tiled, K, N, a_q, a_d, M)
    assert qmm.qmm_device_status() == RANGE, what
    assert qmm.qmm_device_status() == 0                      # the read clears it
    y = gpu_matmul(type_, tiled, K, N, a_q, a_d, M, path=2).cpu().numpy()
    assert qmm.qmm_device_status() == 0
    assert_within_bound(y, y_ref, bound, f"exact path, {what}")


@pytest.mark.parametrize("type_", FOLD_TYPES)
def test_fold_reports_token_row_it_cannot_represent(torch, orc, type_):
    # Row 9 holds a block of 1e5 (the row takes the power-of-two shift) and blocks of about 1e-4, whose
    # fp16 scales (subnormal) lose bits when shifted.  Weight rows 0..79 are zero under the large block,
    # so their outputs come from the small blocks alone: lost bits there would be far above the bound.
    K, N, M = 1024, 160, 140
    x = synth.activations(M, K, seed=53)
    x[9, :32] = np.float32(1e5) * np.sign(x[9, :32])
    x[9, 32:] *= np.float32(1e-4)
    w = synth.weights(N, K, seed=54)
    w[:80, :32] = 0.0
    _range_case(torch, orc, type_, w, x, "token row")


@pytest.mark.parametrize("type_", FOLD_TYPES)
def test_fold_reports_weight_row_it_cannot_represent(torch, orc, type_):
    # Weight row 7: one block large enough for the row shift, the others with subnormal fp16 scales that
    # lose bits when shifted; token rows 0..59 are zero under the large block.
    K, N, M = 1024, 96, 130
    w = synth.weights(N, K, seed=55)
    w[7, :32] *= np.float32(1e6)
    w[7, 32:] *= np.float32(7e-5)
    x = synth.activations(M, K, seed=56)
    x[:60, :32] = 0.0
    _range_case(torch, orc, type_, w, x, "weight row")


def test_fold_matches_exact_kernel(torch, orc):
    # the folded-scale and exact-integer kernels compute the same sum: both within the bound and
    # close to each other
    from tests.gpu_util import gpu_matmul

    w = synth.weights(384, 2048, seed=47)
    x = synth.activations(200, 2048, seed=48, outliers=True)
    _, tiled = gpu_prepare_weight("q4_0", w)
    a_q, a_d = gpu_quantize_act(x)
    y_exact = gpu_matmul("q4_0", tiled, 2048, 384, a_q, a_d, 200, path=2).cpu().numpy()
    y_fold = gpu_matmul_ws("q4_0", tiled, 2048, 384, a_q, a_d, 200).cpu().numpy()
    scale = np.abs(y_exact).max()
    assert np.abs(y_exact - y_fold).max() <= 1e-5 * scale


@pytest.mark.parametrize("scale", [1.0, 5e4])
def test_fold_token_split_is_exact(torch, scale):
    # White-box check of the token preparation: after qmm_matmul_ws the workspace holds, per
    # activation element, two fp16 numbers hi, lo with hi = fp16(v) (nearest) and hi + lo == v
    # exactly, v = d_a * q_a * 2^-s, where 2^s (stored per token row) is 1 unless the row's range
    # needs the shift.  Region offsets follow GemmWsLayout in qmm_internal.cuh.
    import block_quantized_matmul_gb300 as qmm

    M, K, N = 200, 1024, 128
    x = synth.activations(M, K, seed=51, outliers=True)
    x[7] *= np.float32(scale)
    w = synth.weights(N, K, seed=52)
    _, tiled = gpu_prepare_weight("q4_0", w)
    a_q, a_d = gpu_quantize_act(x)
    nbytes = qmm.matmul_workspace_size(M, K)
    ws = torch.full((nbytes + 256,), 0x5A, dtype=torch.uint8, device="cuda")
    off = (-ws.data_ptr()) % 256
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    qmm.qmm_matmul_ws("q4_0", tiled, K, N, a_q, a_d, M, y, N, ws.data_ptr() + off, nbytes)
    torch.cuda.synchronize()
    buf = ws[off:off + nbytes].cpu().numpy()

    def r256(v):
        return (v + 255) // 256 * 256

    nkt, m_pad, mk2 = K // 32, (M + 7) // 8 * 8, M * K * 2
    lo_off = r256(mk2)
    ts_off = lo_off + r256(mk2) + r256(nkt * m_pad * 2) + r256(nkt * m_pad * 4)
    hi = buf[:mk2].view(np.float16).reshape(M, K)
    lo = buf[lo_off:lo_off + mk2].view(np.float16).reshape(M, K)
    ts = buf[ts_off:ts_off + 4 * M].view(np.float32).astype(np.float64)
    q = a_q.cpu().numpy().astype(np.float64)
    d = np.repeat(a_d.cpu().numpy().view(np.float16).astype(np.float64), 32, axis=1)
    v = d * q / ts[:, None]                                   # exact in float64
    assert np.array_equal(hi, v.astype(np.float16))           # nearest fp16
    assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), v)
    shifted = np.nonzero(ts != 1.0)[0].tolist()
    assert shifted == ([7] if scale > 1 else [])

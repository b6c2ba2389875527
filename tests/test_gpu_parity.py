"""GPU parity: the CUDA path (libqmm through the C ABI) against the CPU oracle on the same seeded inputs.

Bit-exact for the byte work (weight quantization, repack, unpack, activation quantization); for the
fp32 outputs |gpu - oracle| <= 1e-5 * sum_k |w_k * x_k| + 1e-6 per element, the oracle's fp64 value
and bound computed from the oracle's own tiles and activation quants.
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import (TYPES, assert_within_bound, dev_u8, gpu_matmul, gpu_prepare_weight, gpu_quantize_act,
                            torch_mod)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _special_weights(K):
    """Rows that hit the quantizers' corner cases."""
    rows = [np.zeros(K, np.float32)]                                   # all-zero blocks
    r = np.zeros(K, np.float32); r[::32] = 1.0; rows.append(r)         # one non-zero per block
    r = np.full(K, 0.5, np.float32); r[1::2] = -0.5; rows.append(r)    # tie on the max magnitude
    r = np.linspace(-1, 1, K, dtype=np.float32); rows.append(r)
    r = np.full(K, 1e-30, np.float32); rows.append(r)                  # tiny scale (fp16 underflow)
    r = np.full(K, 1e6, np.float32); r[::3] *= -1; rows.append(r)      # Q4_0 fp16 scale overflows to inf
    return np.stack(rows)


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("N,K", [(33, 96), (64, 256), (6, 64)])
def test_quantize_weight_and_repack_bit_exact(torch, orc, type_, N, K):
    w = synth.weights(N, K, seed=N * 7 + K)
    if N == 6:
        w = _special_weights(K)
    flat_d, tiled_d = gpu_prepare_weight(type_, w)
    flat_ref = orc.quantize_rows(type_, w)
    tiled_ref = orc.repack(type_, flat_ref, K, N)
    assert np.array_equal(flat_d.cpu().numpy(), flat_ref.reshape(-1)), "quantize_weight"
    assert np.array_equal(tiled_d.cpu().numpy(), tiled_ref), "repack"


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("N,K", [(1, 32), (33, 64), (100, 320), (4096 + 5, 128)])
def test_repack_unpack_random_bytes(torch, orc, type_, N, K):
    import block_quantized_matmul_gb300 as qmm

    rng = np.random.default_rng(N + K)
    flat = rng.integers(0, 256, size=qmm.flat_size(type_, K, N), dtype=np.uint8)
    flat_d = dev_u8(flat)
    tiled_d = torch.full((qmm.tiled_size(type_, K, N),), 0x5A, dtype=torch.uint8, device="cuda")
    qmm.qmm_repack(type_, flat_d, K, N, tiled_d)
    ref = orc.repack(type_, flat.reshape(N, -1), K, N)
    assert np.array_equal(tiled_d.cpu().numpy(), ref)
    back = torch.zeros_like(flat_d)
    qmm.qmm_unpack(type_, tiled_d, K, N, back)
    assert np.array_equal(back.cpu().numpy(), flat)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 4096), (17, 320), (512, 4096)])
def test_quantize_act_bit_exact(torch, orc, M, K):
    x = synth.activations(M, K, seed=M + K, outliers=True)
    a_q, a_d = gpu_quantize_act(x)
    q_ref, d_ref = orc.quantize_act(x)
    assert np.array_equal(a_q.cpu().numpy(), q_ref)
    assert np.array_equal(a_d.cpu().numpy().view(np.uint16), d_ref)


def test_quantize_act_special_blocks_and_strides(torch, orc):
    import block_quantized_matmul_gb300 as qmm

    K = 256
    x = np.zeros((4, K), np.float32)
    x[0, :32] = [127, 2.5, -2.5, 63.5, -63.5, 0.4, -0.5, 1.5] + [0] * 24      # exact ties
    x[1, 32:64] = 1e-40                                                       # subnormal amax
    x[2, 64:96] = np.float32(3e38)                                             # huge values
    x[3] = synth.activations(1, K, seed=5)[0]
    q_ref, d_ref = orc.quantize_act(x)
    # strided rows (ldx > K) and an unaligned base pointer (scalar-load path)
    for ldx, off in [(K, 0), (K + 4, 0), (K + 3, 1)]:
        buf = np.zeros(4 * ldx + off + 4, np.float32)
        for m in range(4):
            buf[off + m * ldx: off + m * ldx + K] = x[m]
        xd = torch.from_numpy(buf).cuda()
        a_q = torch.full((4, K), 99, dtype=torch.int8, device="cuda")
        a_d = torch.full((4, K // 32), 0x7E00, dtype=torch.int16, device="cuda")
        qmm.qmm_quantize_act(xd.data_ptr() + 4 * off, 4, K, ldx, a_q, a_d)
        torch.cuda.synchronize()
        assert np.array_equal(a_q.cpu().numpy(), q_ref), (ldx, off)
        assert np.array_equal(a_d.cpu().numpy().view(np.uint16), d_ref), (ldx, off)


def _parity_case(torch, orc, type_, N, K, M, path, outliers=False, ldy=None):
    w = synth.weights(N, K, seed=3 * N + K)
    x = synth.activations(M, K, seed=M * 11 + K, outliers=outliers)
    flat_ref = orc.quantize_rows(type_, w)
    tiled_ref = orc.repack(type_, flat_ref, K, N)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
    _, tiled_d = gpu_prepare_weight(type_, w)
    assert np.array_equal(tiled_d.cpu().numpy(), tiled_ref)
    a_q, a_d = gpu_quantize_act(x)
    y = gpu_matmul(type_, tiled_d, K, N, a_q, a_d, M, path=path, ldy=ldy).cpu().numpy()
    assert_within_bound(y[:, :N], y_ref, bound, f"{type_} N={N} K={K} M={M} path={path}")
    if ldy is not None and ldy > N:
        assert np.isnan(y[:, N:]).all(), "columns past N must stay untouched"
    return y


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 16, 17])
@pytest.mark.parametrize("N,K", [(100, 256), (33, 1056), (300, 4096)])
def test_matvec_parity(torch, orc, type_, M, N, K):
    _parity_case(torch, orc, type_, N, K, M, path=1)


@pytest.mark.parametrize("type_", TYPES)
def test_matvec_ragged_and_ldy(torch, orc, type_):
    _parity_case(torch, orc, type_, 1, 32, 1, path=1)          # one row, one tile
    _parity_case(torch, orc, type_, 31, 64, 3, path=1, ldy=40)  # ldy > N
    _parity_case(torch, orc, type_, 65, 32 * 37, 5, path=1, outliers=True)


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 4, 16])
def test_matvec_k_passes(torch, orc, type_, M):
    """K long enough that the staged activations take several passes that add into y."""
    _parity_case(torch, orc, type_, 70, 32 * 1100, M, path=1)


def test_matvec_is_deterministic(torch, orc):
    w = synth.weights(512, 4096, seed=1)
    x = synth.activations(4, 4096, seed=2)
    _, tiled = gpu_prepare_weight("q4_0", w)
    a_q, a_d = gpu_quantize_act(x)
    y1 = gpu_matmul("q4_0", tiled, 4096, 512, a_q, a_d, 4, path=1)
    y2 = gpu_matmul("q4_0", tiled, 4096, 512, a_q, a_d, 4, path=1)
    assert torch.equal(y1, y2)


# Full-size workloads: the whole output on the GPU, a sample of it in the oracle (every column tile
# at least once, plus both ends), launched exactly as the benchmark launches them.
FULL = [("q4_0", 4096, 4096, 1), ("q8_0", 4096, 14336, 1), ("iq4_nl", 4096, 4096, 8), ("q8_0", 4096, 128256, 1),
        ("mxfp4", 4096, 14336, 1), ("q4_1", 4096, 14336, 1)]


@pytest.mark.parametrize("type_,K,N,M", FULL, ids=lambda v: str(v))
def test_full_size_sampled(torch, orc, type_, K, N, M):
    w = synth.weights(N, K)
    x = synth.activations(M, K)
    flat_ref = orc.quantize_rows(type_, w)
    tiled_ref = orc.repack(type_, flat_ref, K, N)
    del flat_ref
    q_ref, d_ref = orc.quantize_act(x)
    _, tiled_d = gpu_prepare_weight(type_, w)
    del w
    # compare the tiled weight bit for bit in slices (no full host copy of the GPU buffer needed)
    step = 1 << 26
    for s in range(0, tiled_ref.size, step):
        assert np.array_equal(tiled_d[s:s + step].cpu().numpy(), tiled_ref[s:s + step]), f"tiles @ {s}"
    a_q, a_d = gpu_quantize_act(x)
    assert np.array_equal(a_q.cpu().numpy(), q_ref) and np.array_equal(a_d.cpu().numpy().view(np.uint16), d_ref)
    y = gpu_matmul(type_, tiled_d, K, N, a_q, a_d, M, path=0).cpu().numpy()
    rng = np.random.default_rng(0)
    n_ct = (N + 31) // 32
    ns = np.concatenate([np.arange(n_ct) * 32 + rng.integers(0, 32, n_ct), [0, N - 1]]).clip(0, N - 1)
    ms = rng.integers(0, M, ns.size)
    ys, bs = orc.matmul_at(type_, tiled_ref, K, q_ref, d_ref, ms, ns)
    assert_within_bound(y[ms, ns], ys, bs, f"{type_} {K}x{N} M={M}")
    assert np.isfinite(y).all()


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("M", [1, 8, 40])
def test_column_shards_match_the_full_product(torch, orc, type_, M):
    """A rank's contiguous range of column tiles is itself a tiled weight: its product, written at
    column n0 with the full ldy, equals those columns of the full product bit for bit."""
    from block_quantized_matmul_gb300 import shard

    K, N = 320, 200
    w = synth.weights(N, K, seed=21)
    x = synth.activations(M, K, seed=22)
    _, tiled = gpu_prepare_weight(type_, w)
    a_q, a_d = gpu_quantize_act(x)
    full = gpu_matmul(type_, tiled, K, N, a_q, a_d, M, path=0)
    import block_quantized_matmul_gb300 as qmm

    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    for r in range(3):
        sh = shard.shard(type_, K, N, r, 3)
        if sh.n_local:
            qmm.qmm_matmul(type_, tiled[sh.byte_offset:], K, sh.n_local, a_q, a_d, M, y[:, sh.n0:], N)
    torch.cuda.synchronize()
    assert torch.equal(y, full)


def test_quantize_act_golden_cases(torch):
    """The hand-worked blocks of tests/golden/act_quant_cases.txt through the GPU quantizer, against
    the worked-out codes and scales directly."""
    import block_quantized_matmul_gb300 as qmm
    from tests.test_oracle import _read_act_cases

    cases = _read_act_cases()
    x = np.stack([c[1] for c in cases])
    M = x.shape[0]
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    a_q = torch.full((M, 32), 99, dtype=torch.int8, device="cuda")
    a_d = torch.full((M, 1), 0x7E00, dtype=torch.int16, device="cuda")
    qmm.qmm_quantize_act(xd, M, 32, 32, a_q, a_d)
    torch.cuda.synchronize()
    q = a_q.cpu().numpy()
    d = a_d.cpu().numpy().view(np.uint16)[:, 0]
    for i, (name, _, q_exp, d_exp) in enumerate(cases):
        assert np.array_equal(q[i], q_exp), name
        assert d[i] == d_exp, name

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


# Rows in page-locked host memory take the cluster-shared staging: each CTA of a cluster reads and
# quantizes a share of the blocks and stores the records into every CTA of the cluster.  Shapes: a
# grid smaller than one cluster of the largest size, a grid that is not a multiple of the cluster
# size, the headline grid, the narrow (two CTAs per SM) grid, K in several passes, and fewer blocks
# than CTAs in a cluster (K = 64: most CTAs have no share to stage).
HOST_SHAPES = [(300, 1024), (4096, 4096), (14336, 4096), (40000, 256), (100, 33024), (300, 64)]


@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("N,K", HOST_SHAPES)
def test_fused_host_rows_equal_device_rows(torch, orc, type_, N, K):
    """The same bits as the call on device rows, for 1 to 4 tokens (the int8 path), and within the
    oracle's bound where the oracle is quick."""
    import block_quantized_matmul_gb300 as qmm

    w = synth.weights(N, K, seed=N + 3 * K)
    _, tiled = gpu_prepare_weight(type_, w)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N) if N * K <= 4_000_000 else None
    del w
    for M in (1, 2, 3, 4):
        x = synth.activations(M, K, seed=5 * M + K, outliers=M == 3)
        y_dev = gpu_matmul_f32(type_, tiled, K, N, x)
        x_host = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
        y_host = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
        qmm.qmm_matmul_f32(type_, tiled, K, N, x_host, K, M, y_host, N)
        torch.cuda.synchronize()
        assert torch.equal(y_host, y_dev.cpu()), f"host rows differ from device rows: {type_} {N}x{K} M={M}"
        # the workspace variant: one copy of the rows over the link, then the device-row kernel
        ws_bytes = qmm.matmul_f32_workspace_size(M, K)
        ws = torch.full((ws_bytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
        y_ws = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
        qmm.qmm_matmul_f32_ws(type_, tiled, K, N, x_host, K, M, y_ws, N, ws, ws_bytes)
        torch.cuda.synchronize()
        assert torch.equal(y_ws, y_dev.cpu()), f"workspace call differs: {type_} {N}x{K} M={M}"
        assert torch.equal(ws[: M * K].view(M, K).cpu(), x_host), "the workspace holds the rows"
        if tiled_ref is not None:
            q_ref, d_ref = orc.quantize_act(x)
            y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
            assert_within_bound(y_host.numpy(), y_ref, bound, f"host rows {type_} {N}x{K} M={M}")


@pytest.mark.parametrize("type_", ["q4_0", "iq4_nl"])
def test_fused_host_rows_strided_unaligned(torch, type_):
    """Host rows with an odd stride that start one float past a 16-byte boundary (scalar loads)."""
    import block_quantized_matmul_gb300 as qmm

    K, N, M, ldx = 2048, 1000, 4, 2051
    w = synth.weights(N, K, seed=77)
    _, tiled = gpu_prepare_weight(type_, w)
    x = synth.activations(M, K, seed=78)
    y_dev = gpu_matmul_f32(type_, tiled, K, N, x)
    buf = torch.full((1 + M * ldx,), float("nan"), dtype=torch.float32).pin_memory()
    rows = buf[1:].view(M, ldx)
    rows[:, :K] = torch.from_numpy(np.ascontiguousarray(x))
    y_host = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    qmm.qmm_matmul_f32(type_, tiled, K, N, rows, ldx, M, y_host, N)
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu())
    ws_bytes = qmm.matmul_f32_workspace_size(M, K)
    ws = torch.zeros(ws_bytes // 4, dtype=torch.float32, device="cuda")
    y_ws = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_matmul_f32_ws(type_, tiled, K, N, rows, ldx, M, y_ws, N, ws, ws_bytes)
    torch.cuda.synchronize()
    assert torch.equal(y_ws, y_dev)


@pytest.mark.parametrize("M", [1, 4, 9])
def test_fused_ws_device_rows_leave_the_workspace_alone(torch, M):
    """Device rows need no copy: the workspace variant runs the plain call and never writes it."""
    import block_quantized_matmul_gb300 as qmm

    K, N = 1024, 700
    w = synth.weights(N, K, seed=91)
    _, tiled = gpu_prepare_weight("q8_0", w)
    x = synth.activations(M, K, seed=92)
    y_dev = gpu_matmul_f32("q8_0", tiled, K, N, x)
    ws_bytes = qmm.matmul_f32_workspace_size(M, K)
    ws = torch.full((ws_bytes // 4,), 7.0, dtype=torch.float32, device="cuda")
    y_ws = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_matmul_f32_ws("q8_0", tiled, K, N, torch.from_numpy(x).cuda(), K, M, y_ws, N, ws, ws_bytes)
    torch.cuda.synchronize()
    assert torch.equal(y_ws, y_dev)
    assert bool((ws == 7.0).all())


def test_fused_ws_host_rows_back_to_back(torch):
    """Consecutive calls on one workspace and stream, each with new host rows: every call's copy waits
    for the decode kernel before it, so no call reads rows of another."""
    import block_quantized_matmul_gb300 as qmm

    K, N, M, calls = 4096, 4096, 1, 24
    w = synth.weights(N, K, seed=93)
    _, tiled = gpu_prepare_weight("q4_0", w)
    xs = [synth.activations(M, K, seed=100 + c) for c in range(calls)]
    refs = [gpu_matmul_f32("q4_0", tiled, K, N, x).cpu() for x in xs]
    ws_bytes = qmm.matmul_f32_workspace_size(M, K)
    ws = torch.empty(ws_bytes // 4, dtype=torch.float32, device="cuda")
    x_host = [torch.from_numpy(x).pin_memory() for x in xs]
    y_host = [torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory() for _ in xs]
    for c in range(calls):
        qmm.qmm_matmul_f32_ws("q4_0", tiled, K, N, x_host[c], K, M, y_host[c], N, ws, ws_bytes)
    torch.cuda.synchronize()
    for c in range(calls):
        assert torch.equal(y_host[c], refs[c]), f"call {c}"


def test_fused_refuses_pageable_host_memory(torch):
    """x or y in pageable host memory is refused (INVALID_ARG) before anything is enqueued."""
    import block_quantized_matmul_gb300 as qmm

    K, N, M = 256, 64, 1
    _, tiled = gpu_prepare_weight("q8_0", synth.weights(N, K, seed=5))
    x_page = torch.from_numpy(synth.activations(M, K, seed=6))
    assert not x_page.is_pinned()
    x_dev = x_page.cuda()
    y_dev = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    y_page = torch.full((M, N), float("nan"), dtype=torch.float32)
    ws_bytes = qmm.matmul_f32_workspace_size(M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    calls = [lambda: qmm.qmm_matmul_f32("q8_0", tiled, K, N, x_page, K, M, y_dev, N),
             lambda: qmm.qmm_matmul_f32("q8_0", tiled, K, N, x_dev, K, M, y_page, N),
             lambda: qmm.qmm_matmul_f32_ws("q8_0", tiled, K, N, x_page, K, M, y_dev, N, ws, ws_bytes),
             lambda: qmm.qmm_matmul_f32_ws("q8_0", tiled, K, N, x_dev, K, M, y_page, N, ws, ws_bytes)]
    for call in calls:
        with pytest.raises(qmm.QmmError) as e:
            call()
        assert e.value.status == 1
    torch.cuda.synchronize()
    assert bool(torch.isnan(y_dev).all()) and bool(torch.isnan(y_page).all())


@pytest.mark.parametrize("type_", ["q8_0", "iq4_nl"])
@pytest.mark.parametrize("M", [9, 17])
def test_fused_ws_host_rows_many_tokens(torch, orc, type_, M):
    """Host rows for the fp16 mma decode (9 tokens) and for more rows than one decode launch takes (17:
    a 16-row group, then one row): the rows are copied once, every group reads the device copy."""
    import block_quantized_matmul_gb300 as qmm

    K, N = 2048, 520
    w = synth.weights(N, K, seed=95)
    _, tiled = gpu_prepare_weight(type_, w)
    x = synth.activations(M, K, seed=96)
    y_dev = gpu_matmul_f32(type_, tiled, K, N, x)
    x_host = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    y_host = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    ws_bytes = qmm.matmul_f32_workspace_size(M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    qmm.qmm_matmul_f32_ws(type_, tiled, K, N, x_host, K, M, y_host, N, ws, ws_bytes)
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu())
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul(type_, orc.repack(type_, orc.quantize_rows(type_, w), K, N), K, N, q_ref, d_ref)
    assert_within_bound(y_host.numpy(), y_ref, bound, f"workspace call, host rows {type_} M={M}")

"""qmm_matmul_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (custom allocators or memory pools that must not see foreign allocations, runtimes that
pre-plan all device memory, allocation-free critical sections) get the tensor-core path with its
workspace in the library's fixed per-device scratch array.  This file is collected last on purpose.
The test calls the C ABI (through the binding) twice in a row with different inputs -- the second
call runs on scratch left dirty by the first.  Each result must equal that of the existing workspace
entry point, qmm_matmul_ws, bit for bit (the same kernels run on the same inputs), and the oracle's Y
within the tolerance the other parity tests use.
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import assert_within_bound, gpu_matmul_ws, gpu_prepare_weight, gpu_quantize_act, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


def _noalloc(torch, type_, tiled, K, N, a_q, a_d, M):
    import block_quantized_matmul_gb300 as qmm

    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_matmul_noalloc(type_, tiled, K, N, a_q, a_d, M, y, N)
    torch.cuda.synchronize()
    assert qmm.qmm_device_status() == 0
    return y


def test_noalloc_matches_workspace_entry_point_twice(torch, orc):
    type_, K, N = "q4_0", 1024, 544
    w = synth.weights(N, K, seed=31)
    tiled_ref = orc.repack(type_, orc.quantize_rows(type_, w), K, N)
    _, tiled = gpu_prepare_weight(type_, w)
    for call, (M, seed) in enumerate([(300, 32), (130, 33)]):        # two calls in a row, different M
        x = synth.activations(M, K, seed=seed, outliers=True)
        a_q, a_d = gpu_quantize_act(x)
        y_na = _noalloc(torch, type_, tiled, K, N, a_q, a_d, M)
        y_ws = gpu_matmul_ws(type_, tiled, K, N, a_q, a_d, M)
        assert torch.equal(y_na, y_ws), f"noalloc differs from the workspace entry point, call {call}"
        q_ref, d_ref = orc.quantize_act(x)
        y_ref, bound = orc.matmul(type_, tiled_ref, K, N, q_ref, d_ref)
        assert_within_bound(y_na.cpu().numpy(), y_ref, bound, f"noalloc vs oracle, call {call}")


def test_noalloc_decode_rows_and_size_limit(torch):
    import block_quantized_matmul_gb300 as qmm

    K, N = 256, 96
    w = synth.weights(N, K, seed=34)
    _, tiled = gpu_prepare_weight("q8_0", w)
    x = synth.activations(4, K, seed=35)
    a_q, a_d = gpu_quantize_act(x)
    y_na = _noalloc(torch, "q8_0", tiled, K, N, a_q, a_d, 4)
    y_ws = gpu_matmul_ws("q8_0", tiled, K, N, a_q, a_d, 4)
    assert torch.equal(y_na, y_ws)
    # a workspace beyond the fixed scratch is refused before anything is launched
    limit = qmm.matmul_noalloc_max_workspace()
    M_big, K_big = 4096, 4096
    assert qmm.matmul_workspace_size(M_big, K_big) > limit
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_matmul_noalloc("q8_0", tiled, K_big, N, a_q, a_d, M_big, y_na, N)
    assert e.value.status == 1

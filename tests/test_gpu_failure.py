"""Failure detection on the GPU without a fault: a bounded pipeline wait runs out on purpose.

qmm_selftest_timeout launches one CTA that waits, through the pipelined kernels' own bounded-wait
helper, for a barrier phase that nothing completes.  The wait gives up after its limit, raises the
CTA's abort flag (a second waiter with the normal limit must then give up at once) and sets the
device status word; the host reads QMM_ERR_TIMEOUT, and the context keeps working.
"""
import time

import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth
from tests.gpu_util import (assert_within_bound, gpu_matmul, gpu_matmul_ws, gpu_prepare_weight, gpu_quantize_act,
                            torch_mod)

pytestmark = pytest.mark.gpu
TIMEOUT = 5


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    return t


@pytest.mark.parametrize("unit", [0, 1, 2], ids=["decode_wait", "gemm_wait", "fold_gemm_wait"])
def test_wait_runs_out_and_is_reported(torch, orc, unit):
    import block_quantized_matmul_gb300 as qmm

    assert qmm.qmm_device_status() == 0
    flags = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    qmm.qmm_selftest_timeout(unit, 100_000_000, flags)          # 100 ms
    status = qmm.qmm_device_status()                             # synchronizes
    elapsed = time.perf_counter() - t0
    assert status == TIMEOUT
    assert flags.cpu().tolist() == [0, 0], "both waits must give up"
    # the second waiter (2 s limit) gave up on the abort flag, well before its own limit
    assert 0.09 < elapsed < 1.5, elapsed
    assert qmm.qmm_device_status() == 0, "reading the status clears it"
    # the context still runs the hot path correctly
    K, N, M = 512, 96, 3 if unit == 0 else 40
    w = synth.weights(N, K, seed=unit)
    x = synth.activations(M, K, seed=unit + 1)
    q_ref, d_ref = orc.quantize_act(x)
    y_ref, bound = orc.matmul("q4_0", orc.repack("q4_0", orc.quantize_rows("q4_0", w), K, N), K, N, q_ref, d_ref)
    _, tiled = gpu_prepare_weight("q4_0", w)
    a_q, a_d = gpu_quantize_act(x)
    if unit == 2:      # the folded-scale GEMM runs on the workspace path
        y = gpu_matmul_ws("q4_0", tiled, K, N, a_q, a_d, M).cpu().numpy()
    else:
        y = gpu_matmul("q4_0", tiled, K, N, a_q, a_d, M, path=0).cpu().numpy()
    assert_within_bound(y, y_ref, bound, "after the timeout")
    assert qmm.qmm_device_status() == 0

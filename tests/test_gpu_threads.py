"""Host threads calling the library at the same time, from the very first call of a fresh process.

The first calls resolve one-time state (the tensor-map encoder, the SM count, per-kernel shared-memory
limits, the cluster occupancy of the host-row decode); several threads doing that at once must all get
a working path.  Each thread runs the GEMM, the decode kernel or the decode on pinned host rows on its
own stream and checks its result against a single-threaded run.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys, threading
    sys.path.insert(0, ROOT)
    import torch
    import block_quantized_matmul_gb300 as qmm
    from block_quantized_matmul_gb300 import synth
    K, N = 1024, 640
    w = torch.from_numpy(synth.weights(N, K, seed=4)).cuda()
    flat = torch.empty(qmm.flat_size("q4_0", K, N), dtype=torch.uint8, device="cuda")
    tiled = torch.empty(qmm.tiled_size("q4_0", K, N), dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(synth.activations(64, K, seed=5)).cuda()
    torch.cuda.synchronize()
    errors, results = [], {}

    def run(i):
        s = torch.cuda.Stream()
        if i % 3 == 2:                           # decode on pinned host rows (cluster-shared staging)
            xh = x[:1].cpu().pin_memory()
            yh = torch.full((1, N), float("nan"), dtype=torch.float32).pin_memory()
            qmm.qmm_matmul_f32("q4_0", tiled, K, N, xh, K, 1, yh, N, stream=s)
            s.synchronize()
            return yh.clone()
        M = 1 + (i % 3) * 63                     # decode (M = 1) and GEMM (M = 64) threads
        a_q = torch.empty((M, K), dtype=torch.int8, device="cuda")
        a_d = torch.empty((M, K // 32), dtype=torch.int16, device="cuda")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        nb = qmm.matmul_workspace_size(M, K)
        ws = torch.empty(nb + 256, dtype=torch.uint8, device="cuda")
        wp = ws.data_ptr() + (-ws.data_ptr()) % 256
        with torch.cuda.stream(s):
            qmm.qmm_quantize_act(x[:M].contiguous(), M, K, K, a_q, a_d, stream=s)
            qmm.qmm_matmul_ws("q4_0", tiled, K, N, a_q, a_d, M, y, N, wp, nb, stream=s)
        s.synchronize()
        return y.cpu()

    def work(i):
        try:
            results[i] = run(i)
        except Exception as exc:
            errors.append(repr(exc))

    qmm.qmm_quantize_weight("q4_0", w, N, K, K, flat)
    qmm.qmm_repack("q4_0", flat, K, N, tiled)
    torch.cuda.synchronize()
    threads = [threading.Thread(target=work, args=(i,)) for i in range(9)]
    for t in threads: t.start()
    for t in threads: t.join()
    assert not errors, errors
    # the same calls once more, one thread: identical bits (both paths are deterministic)
    ref = {k: run(k) for k in range(3)}
    for i in range(9):
        assert torch.equal(results[i], ref[i % 3]), i
    assert torch.equal(ref[2], ref[0])           # host rows: the device-row bits
    assert qmm.qmm_device_status() == 0
    print("threads ok")
""").replace("ROOT", repr(ROOT))


def test_concurrent_first_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_matmul_gb300 import build

    build.build()
    r = subprocess.run([sys.executable, "-c", SCRIPT], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "threads ok" in r.stdout

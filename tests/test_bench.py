"""Host-side checks of bench.py's bookkeeping (no GPU): workload names, the launch count each step
claims, and the recorded-traffic lookup."""
from types import SimpleNamespace

import bench


def _launches(type_, K, N, M, fused, flat=False):
    wl = SimpleNamespace(type_=type_, K=K, N=N, M=M, fused=fused, flat_layout=flat)
    return bench.Workload.launches_per_step(wl)


def test_workload_names():
    assert bench.workload_name("q8_0", 4096, 14336, 1) == "q8_0_matvec_K4096_N14336_M1"
    assert bench.workload_name("iq4_nl", 4096, 4096, 8) == "iq4_nl_matmul_K4096_N4096_M8"
    assert bench.workload_name("q4_0", 4096, 14336, 512) == "q4_0_prefill_gemm_K4096_N14336_M512"
    assert bench.workload_name("q4_0", 4096, 14336, 1, "flat") == "q4_0_flat_matvec_K4096_N14336_M1"
    names = [bench.workload_name(*c) for c in [bench.HEADLINE] + bench.OTHERS]
    assert len(names) == len(set(names))


def test_launches_per_step():
    assert _launches("q8_0", 4096, 14336, 1, fused=True) == 1             # one fused decode kernel
    assert _launches("q8_0", 4096, 14336, 1, fused=False) == 2            # quantize + decode
    assert _launches("iq4_nl", 4096, 4096, 8, fused=False) == 2
    assert _launches("q4_0", 4096, 14336, 512, fused=False) == 3          # quantize + prepare + GEMM
    assert _launches("q4_0", 32 * 1100, 70, 1, fused=True) == 2           # two K passes (1024 blocks each)
    assert _launches("q4_0", 32 * 1100, 70, 16, fused=False) == 1 + 18    # 16 rows: 64 blocks a pass
    assert _launches("q4_0", 4096, 70, 20, fused=False) == 3
    assert _launches("q4_0", 4096, 14336, 1, fused=False, flat=True) == 2  # quantize + flat decode
    assert _launches("q4_0", 32 * 800, 14336, 5, fused=False, flat=True) == 1 + 2 * 3


def test_recorded_traffic_only_for_known_workloads():
    assert bench.recorded_traffic("no_such_workload") is None
    hbm, bf16, src = bench.measured_peaks()
    assert hbm > 0 and bf16 > 0 and src in ("measured", "fallback")
    assert len(bench.kernel_source_hash("matvec")) == 16 and bench.kernel_source_hash("gemm") != bench.kernel_source_hash("matvec")


def test_kernel_families_hash_every_source_they_compile():
    # every CUDA source and private header of the library belongs to the hash of at least one family,
    # so an edit of any of them invalidates the recorded DRAM traffic it could affect
    import glob
    import os

    csrc = os.path.join(os.path.dirname(bench.__file__), "block_quantized_matmul_gb300", "csrc")
    hashed = set(bench.KERNEL_FILES["matvec"]) | set(bench.KERNEL_FILES["gemm"])
    kernels = {"matvec.cu", "gemm_tc.cu", "gemm_fold.cu", "pipeline.cuh", "tc_common.cuh", "qmm_internal.cuh"}
    present = {os.path.basename(p) for p in glob.glob(os.path.join(csrc, "*.cu*"))}
    assert kernels <= present and kernels <= hashed

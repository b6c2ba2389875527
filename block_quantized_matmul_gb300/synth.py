"""Seeded synthetic inputs for the tiled block-32 quantized matmul.

This module only draws random numbers.  It holds none of the quantization, tiling or matmul
arithmetic, so both the CUDA path and the CPU oracle can take their inputs from it.

Workloads (typical LLM projection shapes; no public dataset is involved):
  * weights: fp32 [N, K] (row n holds the K inputs of output n), i.i.d. N(0, 0.02^2);
  * activations: fp32 [M, K], i.i.d. N(0, 1), optionally with 1 % of the entries (uniformly chosen
    positions) multiplied by 20 to model outlier features.

Every generator takes an explicit seed; numpy's PCG64 stream makes the draws identical on x86 and Arm.
"""
from __future__ import annotations

import numpy as np

WEIGHT_SEED = 0
ACT_SEED = 1
OUTLIER_SEED = 2
WEIGHT_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_SCALE = 20.0

# Named workloads: (type, K, N, M list).  N is the number of weight rows (outputs).
WORKLOADS = {
    "q4_0_matvec_4096x4096_b1": ("q4_0", 4096, 4096, [1]),
    "q8_0_matvec_4096x14336_b1": ("q8_0", 4096, 14336, [1]),
    "iq4_nl_matmul_4096x4096_b8": ("iq4_nl", 4096, 4096, [8]),
    "q4_0_prefill_gemm_m512_4096x14336": ("q4_0", 4096, 14336, [512]),
    "q8_0_lmhead_4096x128256_b1_b128": ("q8_0", 4096, 128256, [1, 128]),
}


def weights(N: int, K: int, seed: int = WEIGHT_SEED, std: float = WEIGHT_STD) -> np.ndarray:
    """fp32 [N, K] ~ N(0, std^2)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(std)
    return w


def activations(M: int, K: int, seed: int = ACT_SEED, outliers: bool = False,
                outlier_seed: int = OUTLIER_SEED) -> np.ndarray:
    """fp32 [M, K] ~ N(0, 1); with outliers, 1 % of the entries (chosen by outlier_seed) are x20."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        orng = np.random.Generator(np.random.PCG64(outlier_seed))
        count = max(1, int(round(OUTLIER_FRACTION * M * K)))
        pos = orng.choice(M * K, size=count, replace=False)
        x.reshape(-1)[pos] *= np.float32(OUTLIER_SCALE)
    return x

"""A host model of the folded-scale GEMM's arithmetic, checked against the oracle's exact result.

The model follows the kernel step by step on all-positive data, where every rounding of the
accumulation pushes the same way:
  * dequantized values d*q split exactly into fp16 hi + lo (weights and activations);
  * per K = 16 step, three products (hi*hi, hi*lo, lo*hi), each summed over the 16 K and added
    into an fp32 accumulator with ONE rounding per product (the rounding of the tensor cores'
    accumulation is not documented, so both round-to-nearest and round-toward-zero are modelled);
  * the accumulator holds one chunk of 128 K; the chunk sums are added in fp32, round to nearest.
The result must be within the stated bound |y - oracle| <= 1e-5 * B + 1e-6 for both rounding
models.  The same model without chunking (one accumulator over all of K) breaks the bound under
round-toward-zero at long K: that is why the kernel drains the accumulator every 128 K.
"""
import numpy as np
import pytest

from block_quantized_matmul_gb300 import synth


def _split(v):
    hi = v.astype(np.float16).astype(np.float64)
    return hi, v - hi                                   # lo is exact in fp16 (tests/test_fold_split.py)


def _acc(acc, add, toward_zero):
    exact = acc + add
    r = exact.astype(np.float32)
    if toward_zero:
        over = np.abs(r.astype(np.float64)) > np.abs(exact)
        r[over] = np.nextafter(r[over], np.float32(0))
    return r.astype(np.float64)


def _model(a, w, chunk_k, toward_zero):
    """a [M, K], w [N, K] dequantized values (float64, exact) -> y [M, N] as the kernel forms it."""
    M, K = a.shape
    ah, al = _split(a)
    wh, wl = _split(w)
    steps = K // 16
    # per K = 16 step, the three products summed over the step (exact in float64: 22-bit products)
    prods = []
    for x, z in ((ah, wh), (ah, wl), (al, wh)):
        prods.append(np.einsum("msk,nsk->smn", x.reshape(M, steps, 16), z.reshape(-1, steps, 16)))
    y = np.zeros((M, w.shape[0]))
    per_chunk = chunk_k // 16
    for c0 in range(0, steps, per_chunk):
        acc = np.zeros_like(y)
        for s in range(c0, min(steps, c0 + per_chunk)):
            for pr in prods:
                acc = _acc(acc, pr[s], toward_zero)
        y = _acc(y, acc, False)                         # CUDA-core fp32 add, round to nearest
    return y


def _case(orc, K, M=2, N=8, seed=61):
    w = np.abs(synth.weights(N, K, seed=seed))
    x = np.abs(synth.activations(M, K, seed=seed + 1))
    flat = orc.quantize_rows("q8_0", w)
    wq = orc.dequantize_flat("q8_0", flat, N, K)        # d_w * q exactly
    a_q, a_d = orc.quantize_act(x)
    d = a_d.view(np.float16).astype(np.float64)
    a = a_q.astype(np.float64) * np.repeat(d, 32, axis=1)
    y_ref, bound = orc.matmul("q8_0", orc.repack("q8_0", flat, K, N), K, N, a_q, a_d)
    return a, wq, y_ref, bound


@pytest.mark.parametrize("toward_zero", [False, True], ids=["nearest", "toward_zero"])
def test_chunked_accumulation_meets_the_bound(orc, toward_zero):
    a, w, y_ref, bound = _case(orc, K=16384)
    y = _model(a, w, chunk_k=128, toward_zero=toward_zero)
    err = np.abs(y - y_ref)
    assert (err <= 1e-5 * bound + 1e-6).all(), (err / bound).max()
    assert (err / bound).max() < 5e-6                   # the design's worst-case estimate


def test_unchunked_accumulation_would_not(orc):
    a, w, y_ref, bound = _case(orc, K=16384)
    y = _model(a, w, chunk_k=16384, toward_zero=True)
    assert (np.abs(y - y_ref) / bound).max() > 1e-5

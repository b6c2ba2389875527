"""Helpers for the GPU parity tests: run one workload through the CUDA path (libqmm, via the binding)
and through the CPU oracle, on the same seeded inputs."""
from __future__ import annotations

import os

import numpy as np

TYPES = ["q4_0", "q8_0", "iq4_nl", "mxfp4", "q4_1"]


def torch_mod():
    import torch

    return torch


def dev_u8(a: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).cuda()


def gpu_prepare_weight(type_, w: np.ndarray):
    """fp32 [N, K] -> (flat, tiled) on the GPU through qmm_quantize_weight + qmm_repack."""
    import block_quantized_matmul_gb300 as qmm

    torch = torch_mod()
    N, K = w.shape
    w_d = torch.from_numpy(np.ascontiguousarray(w)).cuda()
    flat = torch.empty(qmm.flat_size(type_, K, N), dtype=torch.uint8, device="cuda")
    tiled = torch.full((qmm.tiled_size(type_, K, N),), 0xA5, dtype=torch.uint8, device="cuda")
    qmm.qmm_quantize_weight(type_, w_d, N, K, K, flat)
    qmm.qmm_repack(type_, flat, K, N, tiled)
    return flat, tiled


def gpu_quantize_act(x: np.ndarray):
    import block_quantized_matmul_gb300 as qmm

    torch = torch_mod()
    M, K = x.shape
    x_d = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    a_q = torch.full((M, K), 99, dtype=torch.int8, device="cuda")
    a_d = torch.full((M, K // 32), 0x7E00, dtype=torch.int16, device="cuda")
    qmm.qmm_quantize_act(x_d, M, K, K, a_q, a_d)
    return a_q, a_d


def gpu_matmul(type_, tiled, K, N, a_q, a_d, M, path=0, ldy=None):
    import block_quantized_matmul_gb300 as qmm

    torch = torch_mod()
    ldy = N if ldy is None else ldy
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_matmul_path(type_, tiled, K, N, a_q, a_d, M, y, ldy, path)
    torch.cuda.synchronize()
    return y


def assert_within_bound(y_gpu: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what=""):
    """|gpu - oracle| <= 1e-5 * sum_k |w_k x_k| + 1e-6, element by element."""
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    tol = 1e-5 * bound + 1e-6
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance, e.g. at {idx.tolist()}: "
                             f"gpu={y_gpu[tuple(idx[0])]}, ref={y_ref[tuple(idx[0])]}, tol={tol[tuple(idx[0])]}")


def gpu_matmul_ws(type_, tiled, K, N, a_q, a_d, M, ldy=None, fill=0x5A):
    """qmm_matmul_ws with a freshly allocated (and deliberately dirty) workspace."""
    import block_quantized_matmul_gb300 as qmm

    torch = torch_mod()
    ldy = N if ldy is None else ldy
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = qmm.matmul_workspace_size(M, K)
    ws = torch.full((nbytes + 256,), fill, dtype=torch.uint8, device="cuda")
    off = (-ws.data_ptr()) % 256
    qmm.qmm_matmul_ws(type_, tiled, K, N, a_q, a_d, M, y, ldy, ws.data_ptr() + off, nbytes)
    torch.cuda.synchronize()
    return y


def gpu_matmul_f32(type_, tiled, K, N, x: np.ndarray, ldx=None, ldy=None, x_offset=0):
    """qmm_matmul_f32 (activation quantization fused into the decode kernel) on fp32 rows x [M, K].
    x is placed in a row-padded device buffer (row stride ldx) starting x_offset floats in."""
    import block_quantized_matmul_gb300 as qmm

    torch = torch_mod()
    M = x.shape[0]
    ldx = K if ldx is None else ldx
    ldy = N if ldy is None else ldy
    buf = torch.full((x_offset + M * ldx,), float("nan"), dtype=torch.float32, device="cuda")
    rows = buf[x_offset:].view(M, ldx)
    rows[:, :K] = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_matmul_f32(type_, tiled, K, N, rows, ldx, M, y, ldy)
    torch.cuda.synchronize()
    return y


def _oracle_at_task(job):
    """One worker's share of oracle_at_parallel: outputs of a few column tiles, re-indexed locally."""
    import oracle as orc

    type_, tiles, K, a_q, a_d, ms, ns = job
    return orc.matmul_at(type_, tiles, K, a_q, a_d, ms, ns)


def oracle_at_parallel(type_, tiled_ref: np.ndarray, K: int, a_q, a_d, ms, ns, workers=None):
    """The oracle's Y[ms[i], ns[i]] and bounds, computed by a pool of processes started with spawn
    (safe after CUDA is initialized).  Each task gets only the contiguous bytes of the column tiles it
    needs (tile_idx = ct * n_k_tiles + kt, so a column tile is one byte range) and its points with
    the column re-indexed into those tiles."""
    import multiprocessing as mp

    import oracle as orc

    ms = np.asarray(ms, dtype=np.int64)
    ns = np.asarray(ns, dtype=np.int64)
    ct_bytes = (K // 32) * orc.tile_bytes(type_)
    cts = ns // 32
    uniq = np.unique(cts)
    workers = workers or max(1, min(16, os.cpu_count() or 1))
    groups = np.array_split(uniq, min(len(uniq), 4 * workers))
    jobs, where = [], []
    for grp in groups:
        sel = np.nonzero(np.isin(cts, grp))[0]
        local = np.searchsorted(grp, cts[sel])
        tiles = np.concatenate([tiled_ref[c * ct_bytes:(c + 1) * ct_bytes] for c in grp])
        jobs.append((type_, tiles, K, a_q, a_d, ms[sel], local * 32 + ns[sel] % 32))
        where.append(sel)
    y = np.empty(ms.size, np.float64)
    b = np.empty(ms.size, np.float64)
    with mp.get_context("spawn").Pool(workers) as pool:
        for sel, (ys, bs) in zip(where, pool.map(_oracle_at_task, jobs)):
            y[sel] = ys
            b[sel] = bs
    return y, b

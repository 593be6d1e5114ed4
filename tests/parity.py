"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle
on the same seeded inputs (all outputs, or sampled rows and column blocks at
full size) and compare element by element.

Tolerance for the forward output (fp32 accumulation, one final fp16
rounding): |y_gpu - y_ref| <= 1e-3 + 4e-3 * |y_ref|, y_ref in fp64 from the
oracle. Dequantised weights must match the oracle bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_weight_quantized_awq_gb300 import Path, awq_path_supported, linear_forward
from bit_weight_quantized_awq_gb300.synthetic import Problem

ATOL = 1e-3
RTOL = 4e-3


def sample_rows(M: int, n: int = 64, seed: int = 0) -> np.ndarray:
    """Up to n distinct rows, always including 0 and M - 1."""
    if M <= n:
        return np.arange(M, dtype=np.int64)
    rng = np.random.default_rng(seed + M)
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], mid])).astype(np.int64)


def column_blocks(N: int, width: int = 256) -> list[tuple[int, int]]:
    """Column ranges (multiples of 8) covering the start, the middle and the
    ragged end of N; the whole of N when it is small."""
    if N <= 3 * width:
        return [(0, N)]
    mid = (N // 2) // 8 * 8
    end0 = max(mid + width, N - width) // 8 * 8
    return [(0, width), (mid, mid + width), (end0, N)]


def oracle_reference(p: Problem, rows=None, cols=None) -> np.ndarray:
    """fp64 y_ref[rows][:, n0:n1] from the oracle on the (sliced) CPU inputs."""
    x = p.x.reshape(-1, p.K).numpy()
    qw, qz, sc = p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy()
    b = None if p.bias is None else p.bias.numpy()
    if cols is not None:
        n0, n1 = cols
        qw = np.ascontiguousarray(qw[:, n0 // 8:n1 // 8])
        qz = np.ascontiguousarray(qz[:, n0 // 8:n1 // 8])
        sc = np.ascontiguousarray(sc[:, n0:n1])
        b = None if b is None else np.ascontiguousarray(b[n0:n1])
    return oracle.forward(x, qw, qz, sc, b, p.group_size, rows=rows)


def assert_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    y_gpu = y_gpu.astype(np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = ATOL + RTOL * np.abs(y_ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.max(err / bound)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outputs outside 1e-3 + 4e-3|y| "
            f"(worst err/bound {worst:.3g}); first at {idx.tolist()}: "
            f"gpu {[y_gpu[tuple(i)] for i in idx]} ref {[y_ref[tuple(i)] for i in idx]}")


def run_path(p_gpu: Problem, path: Path, out=None) -> torch.Tensor:
    return linear_forward(p_gpu.x, p_gpu.qweight, p_gpu.qzeros, p_gpu.scales, p_gpu.bias,
                          p_gpu.group_size, path=path, out=out)


def paths_for(M: int, K: int, N: int, g: int) -> list[Path]:
    """AUTO plus every explicit path that can serve this shape."""
    out = [Path.AUTO]
    for path in (Path.GENERIC, Path.DECODE, Path.PREFILL, Path.DEQUANT_GEMM):
        if awq_path_supported(M, K, N, g, path):
            out.append(path)
    return out


def check_problem(p: Problem, paths=None, full: bool = True, max_rows: int = 64):
    """Runs every requested path on the GPU and compares with the oracle."""
    M, K, N, g = p.M, p.K, p.N, p.group_size
    dev = torch.device("cuda")
    pg = p.to(dev)
    paths = paths if paths is not None else paths_for(M, K, N, g)
    if full:
        rows, blocks = None, [(0, N)]
    else:
        rows, blocks = sample_rows(M, max_rows), column_blocks(N)
    refs = {blk: oracle_reference(p, rows, None if blk == (0, N) else blk) for blk in blocks}
    for path in paths:
        y = run_path(pg, path).reshape(M, N)
        torch.cuda.synchronize()
        y_np = y.cpu().numpy()
        if rows is not None:
            y_np = y_np[rows]
        for (n0, n1), ref in refs.items():
            assert_close(y_np[:, n0:n1], ref, f"{path.name} M={M} K={K} N={N} g={g} cols {n0}:{n1}")

"""Sharded WQLinear on one GPU, and concatenation of packed weights.

The Predibase Lorax "Tensor Parallel Layers" page splits a linear layer
between ranks in two ways: ColumnLinear gives every rank a slice of
out_features (the outputs are concatenated), RowLinear gives every rank a
slice of in_features (the partial products are summed, then the bias is
added once). Fused projections (Q/K/V, gate/up) are several layers'
weights concatenated along out_features.

Here the shards run one after another on one GPU:

* ``split_columns`` / ``column_parallel_forward``: slices of N (whole packed
  words); each slice is an ordinary forward, the outputs are concatenated --
  for a single token without a copy, every shard writing its slice of one
  output (the page's single-token head path).
* ``split_rows`` / ``row_parallel_forward``: group-aligned slices of K; every
  shard adds its fp32 product into one fp32 buffer from inside its kernel's
  epilogue (``awq_linear_forward_rows``, reading its slice of x in place),
  and ``awq_finish_rows`` adds the bias and rounds once.
* ``concat_columns``: packed Q/K/V or gate/up weights joined along N.

Slicing and concatenating weights is data movement done once when a model is
loaded (torch views made contiguous); every product runs in the CUDA
library. Across GPUs, the fp32 buffers of the row shards would be summed by
an all-reduce before ``awq_finish_rows``; this module does not do that.
"""
from __future__ import annotations

import torch

from ._binding import AWQError, Status, awq_finish_rows, awq_linear_forward_rows
from .layer import _check, _ptr, _stream, linear_forward


def split_columns(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor,
                  bias: torch.Tensor | None, parts: int) -> list[tuple]:
    """``parts`` equal slices of out_features, each (qweight, qzeros, scales,
    bias) contiguous. N / parts must be a multiple of 8 (whole packed words)."""
    N = scales.shape[1]
    if parts < 1 or N % (8 * parts) != 0:
        raise ValueError(f"out_features {N} does not split into {parts} slices of whole 8-column words")
    n = N // parts
    w = n // 8
    out = []
    for r in range(parts):
        out.append((qweight[:, r * w:(r + 1) * w].contiguous(), qzeros[:, r * w:(r + 1) * w].contiguous(),
                    scales[:, r * n:(r + 1) * n].contiguous(),
                    None if bias is None else bias[r * n:(r + 1) * n].contiguous()))
    return out


def split_rows(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor, group_size: int,
               parts: int) -> list[tuple]:
    """``parts`` equal, group-aligned slices of in_features, each (qweight,
    qzeros, scales, group_size). With group_size -1 the single group spans
    every slice, so every slice keeps the one row of zeros and scales. A
    slice must hold whole groups and a multiple of 8 rows (so that its part
    of x starts on a 16-byte boundary)."""
    K = qweight.shape[0]
    if parts < 1 or K % parts != 0:
        raise ValueError(f"in_features {K} does not split into {parts} equal slices")
    kp = K // parts
    if kp % 8 != 0:
        raise ValueError("each slice of in_features must be a multiple of 8 rows")
    out = []
    if group_size == -1:
        for r in range(parts):
            out.append((qweight[r * kp:(r + 1) * kp].contiguous(), qzeros.contiguous(), scales.contiguous(), -1))
        return out
    if kp % group_size != 0:
        raise ValueError(f"slices of {kp} rows do not hold whole groups of {group_size}")
    gp = kp // group_size
    for r in range(parts):
        out.append((qweight[r * kp:(r + 1) * kp].contiguous(), qzeros[r * gp:(r + 1) * gp].contiguous(),
                    scales[r * gp:(r + 1) * gp].contiguous(), group_size))
    return out


def concat_columns(layers: list[tuple]) -> tuple:
    """Joins layers (qweight, qzeros, scales, bias) that share in_features and
    group_size along out_features: fused Q/K/V or gate/up weights. A missing
    bias counts as zeros when another layer has one."""
    if not layers:
        raise ValueError("nothing to concatenate")
    K, G = layers[0][0].shape[0], layers[0][1].shape[0]
    for (qw, qz, sc, _) in layers:
        if qw.shape[0] != K or qz.shape[0] != G or sc.shape[0] != G:
            raise ValueError("layers differ in in_features or number of groups")
    qweight = torch.cat([l[0] for l in layers], dim=1).contiguous()
    qzeros = torch.cat([l[1] for l in layers], dim=1).contiguous()
    scales = torch.cat([l[2] for l in layers], dim=1).contiguous()
    if all(l[3] is None for l in layers):
        bias = None
    else:
        bias = torch.cat([l[3] if l[3] is not None else torch.zeros(l[2].shape[1], dtype=l[2].dtype,
                                                                    device=l[2].device)
                          for l in layers]).contiguous()
    return qweight, qzeros, scales, bias


def column_parallel_forward(x: torch.Tensor, shards: list[tuple], group_size: int,
                            out: torch.Tensor | None = None) -> torch.Tensor:
    """The forward of a column-sharded layer: the shards' outputs side by side,
    shape (*x.shape[:-1], N) with N the shards' out_features added up. The
    shards may differ in width (separate heads: Q, K, V, or a vocabulary cut
    into unequal slices); each is (qweight, qzeros, scales, bias).

    A single token (x holds one row): that row of y is contiguous, so each
    shard's kernel writes its own slice of one output directly. The gathered
    tensor is the only one allocated (none when ``out`` is given) and nothing
    is copied afterwards. This is the single-token branch of the
    vocabulary-sharded head on the Predibase Lorax "Tensor Parallel Layers"
    page (TensorParallelHead, Description: for one-token batches the matmul
    and the gather are fused so as to allocate less), applied to WQLinear
    shards. With several rows a shard's part of y is strided, and the
    shards' outputs are concatenated (the page's gather-then-concatenate
    branch), into ``out`` when it is given.
    """
    if not shards:
        raise ValueError("no shards")
    K = shards[0][0].shape[0]
    for (qw, _, _, _) in shards:
        if qw.shape[0] != K:
            raise ValueError("shards differ in in_features")
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} features, the shards hold {K}")
    widths = [qw.shape[1] * 8 for (qw, _, _, _) in shards]
    N = sum(widths)
    M = x.numel() // K
    dev = shards[0][0].device
    if out is None:
        if dev.type != "cuda":
            raise ValueError("the AWQ library runs on CUDA tensors only")
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _check(out, "out", torch.float16, dev)
        if out.numel() != M * N:
            raise ValueError(f"out holds {out.numel()} elements, the gathered output {M * N}")
    y = out.view(M, N)
    if M == 1:
        c0 = 0
        for (qw, qz, sc, b), n in zip(shards, widths):
            # a [1, n] slice of the row: contiguous, 16-byte aligned (c0 is a
            # multiple of 8 halves)
            linear_forward(x, qw, qz, sc, b, group_size, out=y[:, c0:c0 + n])
            c0 += n
    else:
        torch.cat([linear_forward(x, qw, qz, sc, b, group_size).view(M, n)
                   for (qw, qz, sc, b), n in zip(shards, widths)], dim=1, out=y)
    return y.view(*x.shape[:-1], N)


def row_parallel_forward(x: torch.Tensor, shards: list[tuple], bias: torch.Tensor | None,
                         out: torch.Tensor | None = None) -> torch.Tensor:
    """The forward of a row-sharded layer: every shard adds its fp32 product
    of its slice of x into one fp32 buffer, then the bias is added and the
    sum rounded once to fp16."""
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    _check(x, "x", torch.float16, dev)
    K = sum(s[0].shape[0] for s in shards)
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} features, the shards hold {K}")
    N = shards[0][2].shape[1]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    y32 = torch.zeros((M, N), dtype=torch.float32, device=dev)
    stream = _stream(dev)
    k0 = 0
    for (qw, qz, sc, g) in shards:
        for t, name, dt in ((qw, "qweight", torch.int32), (qz, "qzeros", torch.int32),
                            (sc, "scales", torch.float16)):
            _check(t, name, dt, dev)
        kr = qw.shape[0]
        st = awq_linear_forward_rows(_ptr(x2) + 2 * k0, K, _ptr(qw), _ptr(qz), _ptr(sc), _ptr(y32),
                                     M, kr, N, g, stream)
        if st != Status.OK:
            raise AWQError(st, "awq_linear_forward_rows")
        k0 += kr
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    if bias is not None:
        _check(bias, "bias", torch.float16, dev)
    st = awq_finish_rows(_ptr(y32), _ptr(bias), _ptr(out), M, N, stream)
    if st != Status.OK:
        raise AWQError(st, "awq_finish_rows")
    return out.reshape(*x.shape[:-1], N)

"""Torch-facing wrappers: allocate outputs, pass pointers and the current
stream to the C ABI, reshape. No arithmetic happens here. The library works
on the current CUDA device, so the tensors must be on it (select it with
``torch.cuda.set_device`` or ``torch.cuda.device`` when a process drives
several GPUs).

``AWQLinear`` follows the WQLinear contract (Predibase Lorax "AWQ WQLinear"
page): constructor arguments (w_bit, group_size, qweight, qzeros, scales,
bias) from its Signature; the w_bit == 4, shape and divisibility checks from
Description, __init__; forward = flatten x to 2-D, quantised GEMM, bias,
restore the batch shape (Description, forward steps 1-3); a ``weight``
property returning the raw qweight.
"""
from __future__ import annotations

import torch

from ._binding import (AWQError, Path, Status, awq_dequant, awq_dequant_gidx, awq_gidx_sort,
                       awq_linear_forward_gidx, awq_linear_forward_path, awq_linear_forward_sorted, awq_pack,
                       awq_permute_rows, awq_quantize_rtn)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device):
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def linear_forward(x: torch.Tensor, qweight: torch.Tensor, qzeros: torch.Tensor,
                   scales: torch.Tensor, bias: torch.Tensor | None, group_size: int,
                   path: Path = Path.AUTO, out: torch.Tensor | None = None) -> torch.Tensor:
    """y = x . dequant(qweight, qzeros, scales) + bias, shape (*x.shape[:-1], N)."""
    dev = qweight.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    f16, i32 = torch.float16, torch.int32
    # one combined test first (the common case), the detailed checks only to
    # name what is wrong
    if not (x.dtype == f16 and qweight.dtype == i32 and qzeros.dtype == i32 and scales.dtype == f16
            and x.device == dev and qzeros.device == dev and scales.device == dev
            and x.is_contiguous() and qweight.is_contiguous() and qzeros.is_contiguous()
            and scales.is_contiguous()):
        _check(x, "x", f16, dev)
        _check(qweight, "qweight", i32, dev)
        _check(qzeros, "qzeros", i32, dev)
        _check(scales, "scales", f16, dev)
    if bias is not None:
        _check(bias, "bias", f16, dev)
    K, N = qweight.shape[0], qweight.shape[1] * 8
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} input features, qweight has {K}")
    M = x.numel() // K
    if out is None:
        out = torch.empty((M, N), dtype=f16, device=dev)
    else:
        _check(out, "out", f16, dev)
        if out.numel() != M * N:
            raise ValueError("out has the wrong number of elements")
    st = awq_linear_forward_path(x.data_ptr(), qweight.data_ptr(), qzeros.data_ptr(), scales.data_ptr(),
                                 _ptr(bias), out.data_ptr(), M, K, N, group_size, _stream(dev), int(path))
    if st != Status.OK:
        raise AWQError(st, "awq_linear_forward")
    return out.view(*x.shape[:-1], N)


def dequant(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor,
            group_size: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """W [K, N] fp16 = (q - z) * scale per group, rounded once to fp16."""
    dev = qweight.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    _check(qweight, "qweight", torch.int32, dev)
    _check(qzeros, "qzeros", torch.int32, dev)
    _check(scales, "scales", torch.float16, dev)
    K, N = qweight.shape[0], qweight.shape[1] * 8
    if out is None:
        out = torch.empty((K, N), dtype=torch.float16, device=dev)
    else:
        _check(out, "out", torch.float16, dev)
    st = awq_dequant(_ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(out), K, N, group_size,
                     _stream(dev))
    if st != Status.OK:
        raise AWQError(st, "awq_dequant")
    return out


def dequant_gidx(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor,
                 g_idx: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """W [K, N] fp16 with the group of row k read from g_idx[k] (int32 [K])."""
    dev = qweight.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    _check(qweight, "qweight", torch.int32, dev)
    _check(qzeros, "qzeros", torch.int32, dev)
    _check(scales, "scales", torch.float16, dev)
    _check(g_idx, "g_idx", torch.int32, dev)
    K, N, G = qweight.shape[0], qweight.shape[1] * 8, scales.shape[0]
    if out is None:
        out = torch.empty((K, N), dtype=torch.float16, device=dev)
    else:
        _check(out, "out", torch.float16, dev)
    st = awq_dequant_gidx(_ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx), _ptr(out), K, N, G,
                          _stream(dev))
    if st != Status.OK:
        raise AWQError(st, "awq_dequant_gidx")
    return out


def linear_forward_gidx(x: torch.Tensor, qweight: torch.Tensor, qzeros: torch.Tensor,
                        scales: torch.Tensor, g_idx: torch.Tensor, bias: torch.Tensor | None,
                        out: torch.Tensor | None = None) -> torch.Tensor:
    """y = x . W + bias with the group of input row k read from g_idx[k]."""
    dev = qweight.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    for t, name, dt in ((x, "x", torch.float16), (qweight, "qweight", torch.int32),
                        (qzeros, "qzeros", torch.int32), (scales, "scales", torch.float16),
                        (g_idx, "g_idx", torch.int32)):
        _check(t, name, dt, dev)
    if bias is not None:
        _check(bias, "bias", torch.float16, dev)
    K, N, G = qweight.shape[0], qweight.shape[1] * 8, scales.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _check(out, "out", torch.float16, dev)
    st = awq_linear_forward_gidx(_ptr(x2), _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx),
                                 _ptr(bias), _ptr(out), M, K, N, G, _stream(dev))
    if st != Status.OK:
        raise AWQError(st, "awq_linear_forward_gidx")
    return out.reshape(*x.shape[:-1], N)


def gidx_sort(g_idx: torch.Tensor, groups: int) -> torch.Tensor:
    """The row order that makes an act-order g_idx layer (every group holds
    K / G rows) a grouped one: int32 [K] on the CPU, perm[i] = the original
    row of sorted row i (awq_gidx_sort, a host routine of the library)."""
    gi = g_idx.detach().to("cpu", torch.int32).contiguous()
    K = gi.numel()
    perm = torch.empty(K, dtype=torch.int32)
    st = awq_gidx_sort(_ptr(gi), K, groups, _ptr(perm))
    if st != Status.OK:
        raise AWQError(st, "awq_gidx_sort")
    return perm


def prepare_act_order(qweight: torch.Tensor, g_idx: torch.Tensor, groups: int):
    """(qweight_sorted, perm on the weights' device, group_size) for an
    act-order layer: rows sorted by group once, on the GPU."""
    dev = qweight.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    _check(qweight, "qweight", torch.int32, dev)
    K, N = qweight.shape[0], qweight.shape[1] * 8
    perm = gidx_sort(g_idx, groups).to(dev)
    out = torch.empty_like(qweight)
    st = awq_permute_rows(_ptr(qweight), _ptr(perm), _ptr(out), K, N, _stream(dev))
    if st != Status.OK:
        raise AWQError(st, "awq_permute_rows")
    return out, perm, K // groups


def linear_forward_sorted(x: torch.Tensor, perm: torch.Tensor, qweight_sorted: torch.Tensor,
                          qzeros: torch.Tensor, scales: torch.Tensor, bias: torch.Tensor | None,
                          group_size: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """The forward of an act-order layer prepared by prepare_act_order: x's
    columns gathered in perm order, then the grouped forward."""
    dev = qweight_sorted.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    for t, name, dt in ((x, "x", torch.float16), (perm, "perm", torch.int32),
                        (qweight_sorted, "qweight_sorted", torch.int32), (qzeros, "qzeros", torch.int32),
                        (scales, "scales", torch.float16)):
        _check(t, name, dt, dev)
    if bias is not None:
        _check(bias, "bias", torch.float16, dev)
    K, N = qweight_sorted.shape[0], qweight_sorted.shape[1] * 8
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _check(out, "out", torch.float16, dev)
    st = awq_linear_forward_sorted(_ptr(x2), _ptr(perm), _ptr(qweight_sorted), _ptr(qzeros), _ptr(scales),
                                   _ptr(bias), _ptr(out), M, K, N, group_size, _stream(dev))
    if st != Status.OK:
        raise AWQError(st, "awq_linear_forward_sorted")
    return out.reshape(*x.shape[:-1], N)


def pack(codes: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """uint8 codes [R, C] (low 4 bits used) -> int32 [R, C/8], column 8j + i of
    a row in nibble i of word j: the layout of qweight and qzeros."""
    dev = codes.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    _check(codes, "codes", torch.uint8, dev)
    if codes.dim() != 2:
        raise ValueError("codes must be 2-D [rows, cols]")
    R, C = codes.shape
    if out is None:
        out = torch.empty((R, C // 8), dtype=torch.int32, device=dev)
    else:
        _check(out, "out", torch.int32, dev)
    st = awq_pack(_ptr(codes), _ptr(out), R, C, _stream(dev))
    if st != Status.OK:
        raise AWQError(st, "awq_pack")
    return out


def quantize_rtn(W: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor, group_size: int,
                 out: torch.Tensor | None = None) -> torch.Tensor:
    """qweight int32 [K, N/8]: q = clamp(round_half_even(W / s) + z, 0, 15) per
    group, packed -- the inverse of ``dequant`` for the given scales and zeros."""
    dev = W.device
    if dev.type != "cuda":
        raise ValueError("the AWQ library runs on CUDA tensors only")
    _check(W, "W", torch.float16, dev)
    _check(scales, "scales", torch.float16, dev)
    _check(qzeros, "qzeros", torch.int32, dev)
    K, N = W.shape
    if out is None:
        out = torch.empty((K, N // 8), dtype=torch.int32, device=dev)
    else:
        _check(out, "out", torch.int32, dev)
    st = awq_quantize_rtn(_ptr(W), _ptr(scales), _ptr(qzeros), _ptr(out), K, N, group_size,
                          _stream(dev))
    if st != Status.OK:
        raise AWQError(st, "awq_quantize_rtn")
    return out


class AWQLinear(torch.nn.Module):
    """4-bit weight-only quantised linear layer (W4A16), inference only."""

    def __init__(self, w_bit: int, group_size: int, qweight: torch.Tensor, qzeros: torch.Tensor,
                 scales: torch.Tensor, bias: torch.Tensor | None):
        super().__init__()
        if w_bit != 4:
            raise ValueError("only 4-bit weights are supported")
        self.w_bit = w_bit
        self.in_features = qweight.shape[0]
        self.out_features = qweight.shape[1] * 32 // w_bit
        self.group_size = self.in_features if group_size == -1 else group_size
        if self.group_size <= 0 or self.in_features % self.group_size != 0:
            raise ValueError("in_features must be divisible by group_size")
        if self.out_features % (32 // w_bit) != 0:
            raise ValueError("out_features must be divisible by 8")
        G = self.in_features // self.group_size
        if tuple(qzeros.shape) != (G, self.out_features // 8):
            raise ValueError(f"qzeros must have shape {(G, self.out_features // 8)}")
        if tuple(scales.shape) != (G, self.out_features):
            raise ValueError(f"scales must have shape {(G, self.out_features)}")
        if bias is not None and tuple(bias.shape) != (self.out_features,):
            raise ValueError(f"bias must have shape {(self.out_features,)}")
        self.register_buffer("qweight", qweight)
        self.register_buffer("qzeros", qzeros)
        self.register_buffer("scales", scales)
        self.register_buffer("bias", bias)

    @property
    def weight(self) -> torch.Tensor:
        return self.qweight

    @torch.no_grad()
    def forward(self, x: torch.Tensor, path: Path = Path.AUTO) -> torch.Tensor:
        return linear_forward(x, self.qweight, self.qzeros, self.scales, self.bias,
                              self.group_size, path=path)

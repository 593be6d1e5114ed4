"""The allocation-free entry point, awq_linear_forward_decode_noalloc.

It exists for callers that must not have device memory allocated behind
their back -- serving processes that budget all device memory up front, or
frameworks whose caching allocator owns the GPU -- and keeps the decode
kernel's split-K scratch in one array compiled into the library. These tests
call it through the C ABI on calls made back to back (the second call finds
the array as the first one left it) and compare every output with the CPU
oracle on the same seeded inputs, and with the regular entry point,
awq_linear_forward, both within the suite's tolerance (1e-3 + 4e-3 |y|).

This file is named so that pytest collects it last; it passes on its own in
a fresh process as well as after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import bit_weight_quantized_awq_gb300 as awq
import oracle
from bit_weight_quantized_awq_gb300 import Status
from bit_weight_quantized_awq_gb300.build import build
from bit_weight_quantized_awq_gb300.synthetic import make_problem

ATOL, RTOL = 1e-3, 4e-3


def _call(fn, p, y, stream):
    M, K, N = p.M, p.K, p.N
    b = None if p.bias is None else p.bias.data_ptr()
    return fn(p.x.data_ptr(), p.qweight.data_ptr(), p.qzeros.data_ptr(), p.scales.data_ptr(), b,
              y.data_ptr(), M, K, N, p.group_size, stream)


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_on_consecutive_calls(gpu):
    stream = torch.cuda.current_stream().cuda_stream
    cases = [make_problem(4, 4096, 4096, 128, bias=True, seed=31),
             make_problem(16, 4096, 12288, 128, bias=False, seed=32),
             make_problem(1, 1024, 800, 64, bias=True, seed=33)]
    probs = [c.to("cuda") for c in cases]
    refs = [oracle.forward(c.x.numpy(), c.qweight.numpy(), c.qzeros.numpy(), c.scales.numpy(),
                           None if c.bias is None else c.bias.numpy(), c.group_size) for c in cases]
    # back to back: A, A again, then B and C, each checked against the
    # oracle and against the regular entry point on the same inputs
    for i in [0, 0, 1, 2]:
        p = probs[i]
        y_reg = torch.empty((p.M, p.N), dtype=torch.float16, device="cuda")
        y_new = torch.full((p.M, p.N), float("nan"), dtype=torch.float16, device="cuda")
        assert _call(awq.awq_linear_forward_decode_noalloc, p, y_new, stream) == Status.OK
        assert _call(awq.awq_linear_forward, p, y_reg, stream) == Status.OK
        torch.cuda.synchronize()
        new = y_new.double().cpu().numpy()
        reg = y_reg.double().cpu().numpy()
        assert np.all(np.abs(new - refs[i]) <= ATOL + RTOL * np.abs(refs[i])), ("oracle", p.M, p.K, p.N)
        assert np.all(np.abs(new - reg) <= ATOL + RTOL * np.abs(reg)), ("regular", p.M, p.K, p.N)
    assert awq.awq_last_device_status(stream) == Status.OK


def test_noalloc_rejects_what_it_cannot_hold():
    """Host-side checks, made before anything is enqueued (no GPU needed)."""
    build(quiet=True)
    A, B = 0x10000, 0x20000      # aligned stand-ins, never dereferenced here
    fn = awq.awq_linear_forward_decode_noalloc
    # more than 8192 column tiles of 256
    assert fn(A, A, A, A, None, B, 1, 4096, 8192 * 256 + 256, 128, None) == Status.ERR_TOO_LARGE
    # shapes the decode kernel does not take
    assert fn(A, A, A, A, None, B, 17, 4096, 4096, 128, None) == Status.ERR_INVALID_ARG
    assert fn(A, A, A, A, None, B, 1, 4096, 8, -1, None) == Status.ERR_INVALID_ARG
    # the page's shape rules, alignment, and M = 0
    assert fn(A, A, A, A, None, B, 1, 4096, 12, 128, None) == Status.ERR_INVALID_ARG
    assert fn(A + 2, A, A, A, None, B, 1, 4096, 4096, 128, None) == Status.ERR_MISALIGNED
    assert fn(None, None, None, None, None, None, 0, 4096, 4096, 128, None) == Status.OK
    assert "fixed scratch" in awq.awq_status_string(Status.ERR_TOO_LARGE)

"""The bounded-wait timeout path, made to run out on purpose without a GPU
fault (the fault-test build of the library, include/awq_gb300_fault_test.h).

In that build every device-side wait gives up after about 2 ms, and
awq_test_inject_fault(1) makes the TMA producer of CTA 0 of every decode and
prefill launch issue no copy: that CTA's consumers wait on a stage barrier
that never fills (a flag that nothing sets). Each case checks that

  * the faulty call returns AWQ_OK at launch and the kernel ends by itself;
  * awq_last_device_status() then reports AWQ_ERR_TIMEOUT (and resets the
    split-K counters the aborted kernel left behind);
  * the next normal calls on the same stream match the CPU oracle within
    1e-3 + 4e-3 |y|, twice in a row -- which they would not if a counter of
    the aborted call were still non-zero (a finisher would then start
    summing before its contributors had written);
  * the status word is clean again afterwards.

Shapes: a decode call whose tiles are split between CTAs (CTA 0 contributes
to a tile another CTA finishes, so that finisher's wait runs out too); a
prefill call of whole 256-row tiles; a prefill call whose tiles are split
along k (stream-K, summed by the separate sum kernel).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_weight_quantized_awq_gb300 import Path, Status
from bit_weight_quantized_awq_gb300.build import FAULT_LIB, build
from bit_weight_quantized_awq_gb300.synthetic import make_problem

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 4e-3
_P, _I64, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int


@pytest.fixture(scope="module")
def flib(gpu):
    build(quiet=True)
    lib = ctypes.CDLL(FAULT_LIB)
    lib.awq_linear_forward_path.argtypes = [_P] * 6 + [_I64] * 4 + [_P, _INT]
    lib.awq_linear_forward_path.restype = _INT
    lib.awq_last_device_status.argtypes = [_P]
    lib.awq_last_device_status.restype = _INT
    lib.awq_test_inject_fault.argtypes = [_INT]
    lib.awq_test_inject_fault.restype = None
    yield lib
    lib.awq_test_inject_fault(0)


def _forward(lib, p, y, path, stream):
    b = None if p.bias is None else p.bias.data_ptr()
    return lib.awq_linear_forward_path(p.x.data_ptr(), p.qweight.data_ptr(), p.qzeros.data_ptr(),
                                       p.scales.data_ptr(), b, y.data_ptr(), p.M, p.K, p.N, p.group_size,
                                       stream, int(path))


@pytest.mark.parametrize("M,K,N,g,path", [
    (4, 4096, 4096, 128, Path.DECODE),      # split tiles: CTA 0 feeds another CTA's finisher
    (512, 4096, 4096, 128, Path.PREFILL),   # whole 256-row tiles
    (40, 4096, 1024, 128, Path.PREFILL),    # stream-K pieces summed by the sum kernel
])
def test_wait_runs_out_then_next_calls_match_oracle(flib, M, K, N, g, path):
    cpu = make_problem(M, K, N, g, bias=True, seed=M + 300)
    p = cpu.to("cuda")
    ref = oracle.forward(cpu.x.numpy(), cpu.qweight.numpy(), cpu.qzeros.numpy(), cpu.scales.numpy(),
                         cpu.bias.numpy(), g)
    stream = torch.cuda.current_stream().cuda_stream
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert flib.awq_last_device_status(stream) == Status.OK

    flib.awq_test_inject_fault(1)
    try:
        assert _forward(flib, p, y, path, stream) == Status.OK
    finally:
        flib.awq_test_inject_fault(0)
    assert flib.awq_last_device_status(stream) == Status.ERR_TIMEOUT

    for _ in range(2):
        y.fill_(float("nan"))
        assert _forward(flib, p, y, path, stream) == Status.OK
        torch.cuda.synchronize()
        got = y.double().cpu().numpy()
        err = np.abs(got - ref)
        assert np.all(err <= ATOL + RTOL * np.abs(ref)), f"{path.name}: {np.sum(~(err <= ATOL + RTOL * np.abs(ref)))} outputs off"
    assert flib.awq_last_device_status(stream) == Status.OK

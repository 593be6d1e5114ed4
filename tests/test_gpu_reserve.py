"""awq_reserve: scratch sized once per stream, after which no call on that
stream allocates or synchronises (include/awq_gb300.h, awq_reserve).

Checked where it matters: on a fresh stream, right after awq_reserve and
with no warm-up call, a CUDA graph is captured in global capture mode --
in which any cudaMalloc, cudaFree or stream synchronisation made by a call
would end the capture with an error -- holding decode, prefill,
dequantise-then-GEMM and act-order calls. The graph is replayed twice and
every output compared with the CPU oracle (1e-3 + 4e-3 |y|). A call that
needs more scratch than the reservation returns AWQ_ERR_TOO_LARGE and
leaves the reserved areas as they were.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantized_awq_gb300 as awq
from bit_weight_quantized_awq_gb300 import Path, Status, linear_forward
from bit_weight_quantized_awq_gb300.synthetic import make_problem

from parity import assert_close, oracle_reference

pytestmark = pytest.mark.gpu


def _fwd(p, y, stream, path=Path.AUTO):
    b = None if p.bias is None else p.bias.data_ptr()
    return awq.awq_linear_forward_path(p.x.data_ptr(), p.qweight.data_ptr(), p.qzeros.data_ptr(),
                                       p.scales.data_ptr(), b, y.data_ptr(), p.M, p.K, p.N, p.group_size,
                                       stream, path)


def test_reserved_stream_captures_without_allocating(gpu):
    stream = torch.cuda.Stream()
    h = stream.cuda_stream
    cases = [(4, 4096, 4096, 128, Path.AUTO),           # decode, split tiles
             (512, 4096, 2048, 128, Path.AUTO),         # fused prefill, stream-K sum kernel
             (6144, 1024, 1024, 128, Path.AUTO),        # dequantise-then-GEMM window
             (40, 2048, 1024, 64, Path.PREFILL)]        # prefill at small M, every tile split
    probs = [make_problem(M, K, N, g, bias=True, seed=M + 31) for (M, K, N, g, _) in cases]
    # act-order layer: its sorted forward needs the x reorder area
    G = 16
    K_ao, N_ao, M_ao = 2048, 1024, 8
    ao = make_problem(M_ao, K_ao, N_ao, K_ao // G, bias=False, seed=77)
    gen = torch.Generator().manual_seed(5)
    g_idx = (torch.arange(K_ao) // (K_ao // G))[torch.randperm(K_ao, generator=gen)].to(torch.int32)
    with torch.cuda.stream(stream):
        pg = [p.to("cuda") for p in probs]
        ao_g = ao.to("cuda")
        q_sorted, perm, _ = awq.prepare_act_order(ao_g.qweight, g_idx.cuda(), G)
        ys = [torch.full((p.M, p.N), float("nan"), dtype=torch.float16, device="cuda") for p in probs]
        y_ao = torch.full((M_ao, N_ao), float("nan"), dtype=torch.float16, device="cuda")
    stream.synchronize()
    assert awq.awq_reserve(6144, 4096, 4096, awq.RESERVE_SORTED, h) == Status.OK

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="global"):
        for p, y, (_, _, _, _, path) in zip(pg, ys, cases):
            assert _fwd(p, y, h, path) == Status.OK
        assert awq.awq_linear_forward_sorted(ao_g.x.data_ptr(), perm.data_ptr(), q_sorted.data_ptr(),
                                             ao_g.qzeros.data_ptr(), ao_g.scales.data_ptr(), None,
                                             y_ao.data_ptr(), M_ao, K_ao, N_ao, K_ao // G, h) == Status.OK
    refs = [oracle_reference(p) for p in probs]
    ref_ao = oracle.forward_gidx(ao.x.numpy(), ao.qweight.numpy(), ao.qzeros.numpy(), ao.scales.numpy(),
                                 g_idx.numpy(), None)
    for _ in range(2):
        for y in ys + [y_ao]:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        for y, ref, c in zip(ys, refs, cases):
            assert_close(y.cpu().numpy(), ref, f"reserved graph {c}")
        assert_close(y_ao.cpu().numpy(), ref_ao, "reserved graph, act-order")
    assert awq.awq_last_device_status(h) == Status.OK


def test_call_beyond_the_reservation_is_refused(gpu):
    stream = torch.cuda.Stream()
    h = stream.cuda_stream
    assert awq.awq_reserve(16, 4096, 4096, 0, h) == Status.OK
    small = make_problem(4, 4096, 4096, 128, bias=False, seed=3).to("cuda")
    # 127 column tiles: more arrival counters than the reservation holds (it
    # keeps headroom above the 16 tiles asked for, but not that much)
    wide = make_problem(4, 4096, 32512, 128, bias=False, seed=4).to("cuda")
    y_small = torch.empty((4, 4096), dtype=torch.float16, device="cuda")
    y_wide = torch.empty((4, 32512), dtype=torch.float16, device="cuda")
    assert _fwd(wide, y_wide, h) == Status.ERR_TOO_LARGE
    # the sorted forward's reorder area was not reserved
    assert awq.awq_linear_forward_sorted(small.x.data_ptr(), small.qweight.data_ptr(), small.qweight.data_ptr(),
                                         small.qzeros.data_ptr(), small.scales.data_ptr(), None,
                                         y_small.data_ptr(), 4, 4096, 4096, 128, h) == Status.ERR_TOO_LARGE
    # calls within the reservation still run and are right
    assert _fwd(small, y_small, h) == Status.OK
    stream.synchronize()
    cpu = make_problem(4, 4096, 4096, 128, bias=False, seed=3)
    assert_close(y_small.cpu().numpy(), oracle_reference(cpu), "within the reservation")
    # a larger reservation lifts the limit
    assert awq.awq_reserve(16, 4096, 32512, 0, h) == Status.OK
    assert _fwd(wide, y_wide, h) == Status.OK
    assert awq.awq_last_device_status(h) == Status.OK

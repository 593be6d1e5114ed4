"""GPU parity of the g_idx grouping variant (the group of input row k read
from g_idx[k]; the GPTQ "act-order" tuple the Linear Layer Factory page
lists), against the CPU oracle: awq_dequant_gidx bit for bit, and
awq_linear_forward_gidx within |y - y_ref| <= 1e-3 + 4e-3 |y_ref|.

Tables: random assignments, a GPTQ-style permuted floor table (each group
holds group_size rows, scattered), the plain floor table (must equal the
grouped path's dequant bit for bit), and an out-of-range entry (reported
by awq_last_device_status).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_quantized_awq_gb300 import (Status, awq_last_device_status, dequant, dequant_gidx,
                                            linear_forward_gidx)
from bit_weight_quantized_awq_gb300.synthetic import make_problem

from parity import assert_close, column_blocks, sample_rows

pytestmark = pytest.mark.gpu


def _table(kind, K, G, seed):
    rng = np.random.default_rng(seed)
    if kind == "random":
        return rng.integers(0, G, size=K).astype(np.int32)
    floor = (np.arange(K) // (K // G)).astype(np.int32)
    return floor if kind == "floor" else floor[rng.permutation(K)].copy()


@pytest.mark.parametrize("K,N,G,kind", [(4096, 4096, 32, "act_order"), (1024, 800, 16, "random"),
                                        (336, 104, 7, "random"), (64, 8, 1, "floor")])
def test_dequant_gidx_bit_exact(gpu, K, N, G, kind):
    p = make_problem(1, K, N, K // G, seed=K + G)
    t = _table(kind, K, G, seed=K)
    got = dequant_gidx(p.qweight.cuda(), p.qzeros.cuda(), p.scales.cuda(), torch.from_numpy(t).cuda())
    ref = oracle.dequant_gidx(p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), t)
    assert np.array_equal(got.cpu().numpy().view(np.uint16), ref)


def test_floor_table_equals_grouped_dequant(gpu):
    K, N, g = 2048, 512, 128
    p = make_problem(1, K, N, g, seed=3).to("cuda")
    t = torch.arange(K, dtype=torch.int32, device="cuda") // g
    assert torch.equal(dequant_gidx(p.qweight, p.qzeros, p.scales, t), dequant(p.qweight, p.qzeros, p.scales, g))


@pytest.mark.parametrize("M,K,N,G,bias,kind", [
    (16, 1024, 512, 8, True, "act_order"),
    (300, 2048, 1056, 16, False, "random"),
    (1, 512, 256, 4, True, "floor"),
])
def test_forward_gidx_matches_oracle(gpu, M, K, N, G, bias, kind):
    p = make_problem(M, K, N, K // G, bias=bias, seed=M + K)
    t = _table(kind, K, G, seed=M)
    pg = p.to("cuda")
    y = linear_forward_gidx(pg.x, pg.qweight, pg.qzeros, pg.scales, torch.from_numpy(t).cuda(), pg.bias)
    ref = oracle.forward_gidx(p.x.numpy(), p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), t,
                              None if p.bias is None else p.bias.numpy())
    assert_close(y.cpu().numpy(), ref, f"gidx M={M} K={K} N={N} G={G} {kind}")


def test_forward_gidx_full_size_sampled(gpu):
    """A 7B-class projection with an act-order table, sampled rows/columns."""
    M, K, N, G = 2048, 4096, 12288, 32
    p = make_problem(M, K, N, K // G, bias=True, seed=77)
    t = _table("act_order", K, G, seed=5)
    pg = p.to("cuda")
    y = linear_forward_gidx(pg.x, pg.qweight, pg.qzeros, pg.scales, torch.from_numpy(t).cuda(), pg.bias)
    rows = sample_rows(M, 32)
    yc = y.cpu().numpy()[rows]
    for (n0, n1) in column_blocks(N):
        ref = oracle.forward_gidx(p.x.numpy(), np.ascontiguousarray(p.qweight.numpy()[:, n0 // 8:n1 // 8]),
                                  np.ascontiguousarray(p.qzeros.numpy()[:, n0 // 8:n1 // 8]),
                                  np.ascontiguousarray(p.scales.numpy()[:, n0:n1]), t,
                                  np.ascontiguousarray(p.bias.numpy()[n0:n1]), rows=rows)
        assert_close(yc[:, n0:n1], ref, f"gidx full size cols {n0}:{n1}")


def test_out_of_range_group_is_reported(gpu):
    K, N, G = 256, 64, 4
    p = make_problem(1, K, N, K // G, seed=9).to("cuda")
    t = torch.zeros(K, dtype=torch.int32, device="cuda")
    t[17] = G
    W = dequant_gidx(p.qweight, p.qzeros, p.scales, t)
    stream = torch.cuda.current_stream().cuda_stream
    assert awq_last_device_status(stream) == Status.ERR_INVALID_ARG
    assert torch.count_nonzero(W[17]) == 0
    assert awq_last_device_status(stream) == Status.OK          # the status word was cleared


# Act-order layers run on the grouped kernels: rows sorted by group once
# (awq_gidx_sort on the host, awq_permute_rows on the GPU), x's columns
# gathered in that order every call. Compared with the oracle's g_idx
# forward on the original, unsorted weights.
@pytest.mark.parametrize("M,K,N,G,bias", [
    (1, 4096, 4096, 32, False),      # decode kernel
    (16, 1024, 512, 8, True),
    (32, 2048, 1056, 16, True),      # four token tiles, ragged N
    (200, 2048, 1024, 16, False),    # fused tcgen05 kernel, one 256-row tile
    (40, 1088, 4128, 17, True),      # 64-row groups, ragged K and N
])
def test_act_order_sorted_forward_matches_oracle(gpu, M, K, N, G, bias):
    from bit_weight_quantized_awq_gb300 import linear_forward_sorted, prepare_act_order
    p = make_problem(M, K, N, K // G, bias=bias, seed=M + K + 1)
    t = _table("act_order", K, G, seed=M + 3)
    pg = p.to("cuda")
    qs, perm, g = prepare_act_order(pg.qweight, torch.from_numpy(t), G)
    assert g == K // G
    y = linear_forward_sorted(pg.x, perm, qs, pg.qzeros, pg.scales, pg.bias, g)
    ref = oracle.forward_gidx(p.x.numpy(), p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), t,
                              None if p.bias is None else p.bias.numpy())
    assert_close(y.cpu().numpy(), ref, f"act-order sorted M={M} K={K} N={N} G={G}")
    assert awq_last_device_status(torch.cuda.current_stream().cuda_stream) == Status.OK


def test_act_order_sorted_forward_full_size_sampled(gpu):
    """M = 8 on an 11008 x 4096 projection (decode path), M = 2048 on
    4096 x 12288 (fused tcgen05 path) and M = 6144 (dequantise-then-GEMM:
    the sorted rows are put back in their original order while being
    dequantised, x is not gathered), sampled rows and column blocks."""
    from bit_weight_quantized_awq_gb300 import linear_forward_sorted, prepare_act_order
    for (M, K, N, G) in [(8, 11008, 4096, 86), (2048, 4096, 12288, 32),
                         (6144, 2048, 1024, 16)]:   # the last: rows put back while dequantising
        p = make_problem(M, K, N, K // G, bias=True, seed=K)
        t = _table("act_order", K, G, seed=11)
        pg = p.to("cuda")
        qs, perm, g = prepare_act_order(pg.qweight, torch.from_numpy(t), G)
        y = linear_forward_sorted(pg.x, perm, qs, pg.qzeros, pg.scales, pg.bias, g)
        rows = sample_rows(M, 16)
        yc = y.cpu().numpy()[rows]
        for (n0, n1) in column_blocks(N):
            ref = oracle.forward_gidx(p.x.numpy(), np.ascontiguousarray(p.qweight.numpy()[:, n0 // 8:n1 // 8]),
                                      np.ascontiguousarray(p.qzeros.numpy()[:, n0 // 8:n1 // 8]),
                                      np.ascontiguousarray(p.scales.numpy()[:, n0:n1]), t,
                                      np.ascontiguousarray(p.bias.numpy()[n0:n1]), rows=rows)
            assert_close(yc[:, n0:n1], ref, f"act-order M={M} cols {n0}:{n1}")


def test_permuted_rows_and_gathered_columns_are_exact(gpu):
    from bit_weight_quantized_awq_gb300 import prepare_act_order
    K, N, G = 512, 256, 4
    p = make_problem(1, K, N, K // G, seed=31).to("cuda")
    t = _table("act_order", K, G, seed=2)
    qs, perm, _ = prepare_act_order(p.qweight, torch.from_numpy(t), G)
    assert torch.equal(qs, p.qweight[perm.long()])


def test_bad_permutation_entry_is_reported(gpu):
    from bit_weight_quantized_awq_gb300 import linear_forward_sorted
    K, N, g = 256, 64, 64
    p = make_problem(2, K, N, g, seed=5).to("cuda")
    perm = torch.arange(K, dtype=torch.int32, device="cuda")
    perm[100] = K          # outside [0, K): read as a zero activation, reported
    y = linear_forward_sorted(p.x, perm, p.qweight, p.qzeros, p.scales, None, g)
    stream = torch.cuda.current_stream().cuda_stream
    assert awq_last_device_status(stream) == Status.ERR_INVALID_ARG
    x0 = p.x.clone()
    x0[:, 100] = 0
    from bit_weight_quantized_awq_gb300 import linear_forward
    assert torch.equal(y, linear_forward(x0, p.qweight, p.qzeros, p.scales, None, g))
    assert awq_last_device_status(stream) == Status.OK


def test_bad_permutation_entry_is_reported_when_dequantising(gpu):
    from bit_weight_quantized_awq_gb300 import linear_forward_sorted
    M, K, N, g = 6144, 256, 256, 64
    p = make_problem(M, K, N, g, seed=6).to("cuda")
    perm = torch.arange(K, dtype=torch.int32, device="cuda")
    perm[7] = -1
    linear_forward_sorted(p.x, perm, p.qweight, p.qzeros, p.scales, None, g)
    stream = torch.cuda.current_stream().cuda_stream
    assert awq_last_device_status(stream) == Status.ERR_INVALID_ARG
    assert awq_last_device_status(stream) == Status.OK

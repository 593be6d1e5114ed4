"""GPU parity of the sharded layer (Predibase Lorax "Tensor Parallel Layers":
ColumnLinear / RowLinear) on one GPU, against the CPU oracle of the
unsharded layer, within |y - y_ref| <= 1e-3 + 4e-3 |y_ref|: column slices
run as ordinary forwards and are concatenated; row slices add their fp32
products into one buffer inside their kernels (awq_linear_forward_rows, x
read in place with its full row pitch) and awq_finish_rows adds the bias and
rounds once. M covers the decode kernel, the fused prefill kernel and the
dequantise-then-GEMM path.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_quantized_awq_gb300 import Status, awq_finish_rows, awq_linear_forward_rows
from bit_weight_quantized_awq_gb300.shard import (column_parallel_forward, concat_columns, row_parallel_forward,
                                                  split_columns, split_rows)
from bit_weight_quantized_awq_gb300.synthetic import make_problem

from parity import assert_close, column_blocks, oracle_reference, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N,g,parts", [(1, 4096, 4096, 128, 2), (16, 2048, 2048, 128, 4),
                                           (300, 1024, 1024, 64, 2), (24, 512, 768, -1, 2)])
def test_column_parallel(gpu, M, K, N, g, parts):
    p = make_problem(M, K, N, g, bias=True, seed=M + parts)
    pg = p.to("cuda")
    y = column_parallel_forward(pg.x, split_columns(pg.qweight, pg.qzeros, pg.scales, pg.bias, parts), g)
    assert_close(y.cpu().numpy(), oracle_reference(p), f"column-parallel x{parts}")


@pytest.mark.parametrize("M,K,N,g,parts", [(1, 4096, 4096, 128, 2), (16, 4096, 2048, 128, 4),
                                           (300, 2048, 1024, 64, 2), (8, 1024, 512, -1, 4),
                                           (5, 1024, 800, 64, 2)])
def test_row_parallel(gpu, M, K, N, g, parts):
    p = make_problem(M, K, N, g, bias=True, seed=M * 3 + parts)
    pg = p.to("cuda")
    y = row_parallel_forward(pg.x, split_rows(pg.qweight, pg.qzeros, pg.scales, g, parts), pg.bias)
    assert_close(y.cpu().numpy(), oracle_reference(p), f"row-parallel x{parts}")


def test_row_parallel_large_m_sampled(gpu):
    """M = 2048: every shard takes the dequantise-then-GEMM path."""
    M, K, N, g = 2048, 8192, 2048, 128
    p = make_problem(M, K, N, g, bias=True, seed=21)
    pg = p.to("cuda")
    y = row_parallel_forward(pg.x, split_rows(pg.qweight, pg.qzeros, pg.scales, g, 2), pg.bias).cpu().numpy()
    rows = sample_rows(M, 32)
    for blk in column_blocks(N):
        assert_close(y[rows][:, blk[0]:blk[1]], oracle_reference(p, rows, None if blk == (0, N) else blk),
                     f"row-parallel M=2048 cols {blk}")


def test_rows_accumulate_into_y32(gpu):
    """Two calls on the same buffer add up: y32 = 2 x . W, then y = fp16(y32)."""
    M, K, N, g = 4, 1024, 512, 128
    p = make_problem(M, K, N, g, seed=31)
    pg = p.to("cuda")
    y32 = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        assert awq_linear_forward_rows(pg.x.data_ptr(), K, pg.qweight.data_ptr(), pg.qzeros.data_ptr(),
                                       pg.scales.data_ptr(), y32.data_ptr(), M, K, N, g, s) == Status.OK
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert awq_finish_rows(y32.data_ptr(), None, y.data_ptr(), M, N, s) == Status.OK
    assert_close(y.cpu().numpy(), 2 * oracle_reference(p), "accumulate twice")


def test_fused_projection_equals_separate(gpu):
    layers = [make_problem(16, 2048, n, 128, bias=True, seed=n) for n in (2048, 512, 512)]
    qw, qz, sc, b = concat_columns([(l.qweight, l.qzeros, l.scales, l.bias) for l in layers])
    x = layers[0].x.cuda()
    from bit_weight_quantized_awq_gb300 import linear_forward
    y = linear_forward(x, qw.cuda(), qz.cuda(), sc.cuda(), b.cuda(), 128).cpu().numpy()
    ref = np.concatenate([oracle.forward(layers[0].x.numpy(), l.qweight.numpy(), l.qzeros.numpy(),
                                         l.scales.numpy(), l.bias.numpy(), 128) for l in layers], axis=1)
    assert_close(y, ref, "fused q/k/v")


@pytest.mark.parametrize("widths,g", [((4096, 1024, 1024), 128), ((2048, 2048), -1), ((512, 8, 1024), 128)])
def test_single_token_heads_gather_in_place(gpu, widths, g):
    """One token over heads of unequal widths (the vocabulary-sharded head's
    single-token branch): every shard writes its slice of one output. The
    result is bit for bit the concatenation of the separate forwards (the
    same kernels run on the same shapes), within tolerance of the oracle,
    and with a caller's output nothing is allocated by torch."""
    from bit_weight_quantized_awq_gb300 import linear_forward
    K = 4096
    heads = [make_problem(1, K, n, g, bias=(i != 1), seed=40 + i) for i, n in enumerate(widths)]
    x = heads[0].x.cuda()
    shards = [(h.qweight.cuda(), h.qzeros.cuda(), h.scales.cuda(), None if h.bias is None else h.bias.cuda())
              for h in heads]
    separate = torch.cat([linear_forward(x, *s, g) for s in shards], dim=-1)
    out = torch.empty((1, sum(widths)), dtype=torch.float16, device="cuda")
    column_parallel_forward(x, shards, g, out=out)   # library scratch set up before counting
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    y = column_parallel_forward(x, shards, g, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    assert y.data_ptr() == out.data_ptr()
    assert torch.equal(y.view(torch.int16), separate.view(torch.int16))
    ref = np.concatenate([oracle.forward(heads[0].x.numpy(), h.qweight.numpy(), h.qzeros.numpy(), h.scales.numpy(),
                                         None if h.bias is None else h.bias.numpy(), g) for h in heads], axis=1)
    assert_close(y.cpu().numpy(), ref, f"single-token heads {widths}")


def test_single_token_batch_shape_kept(gpu):
    """x of shape [1, 1, K] (one token of a batch): the gathered output keeps
    the leading dimensions."""
    M, K, N, g = 1, 1024, 1024, 128
    p = make_problem(M, K, N, g, bias=True, seed=50)
    pg = p.to("cuda")
    y = column_parallel_forward(pg.x.view(1, 1, K), split_columns(pg.qweight, pg.qzeros, pg.scales, pg.bias, 4), g)
    assert y.shape == (1, 1, N)
    assert_close(y.view(1, N).cpu().numpy(), oracle_reference(p), "single token, 3-D x")


def test_multi_token_heads_into_callers_output(gpu):
    """Several tokens: the shards' outputs are concatenated into the caller's
    tensor, equal bit for bit to the unsharded column order."""
    M, K, g = 12, 2048, 64
    heads = [make_problem(M, K, n, g, bias=True, seed=60 + n) for n in (1024, 256)]
    x = heads[0].x.cuda()
    shards = [(h.qweight.cuda(), h.qzeros.cuda(), h.scales.cuda(), h.bias.cuda()) for h in heads]
    out = torch.empty((M, 1280), dtype=torch.float16, device="cuda")
    y = column_parallel_forward(x, shards, g, out=out)
    assert y.data_ptr() == out.data_ptr()
    from bit_weight_quantized_awq_gb300 import linear_forward
    separate = torch.cat([linear_forward(x, *s, g) for s in shards], dim=-1)
    assert torch.equal(y.view(torch.int16), separate.view(torch.int16))

"""Host-side checks of the sharding helpers (Predibase Lorax "Tensor Parallel
Layers" page: ColumnLinear concatenates the outputs of out_features slices,
RowLinear sums the products of in_features slices before adding the bias
once), with the CPU oracle doing the arithmetic: shard-then-combine must
equal the unsharded layer -- exactly for column slices and concatenation
(every output column is computed the same way), and to fp64 rounding for
row slices (the same terms summed in another grouping).
"""
import numpy as np
import pytest

import oracle
from bit_weight_quantized_awq_gb300.shard import concat_columns, split_columns, split_rows
from bit_weight_quantized_awq_gb300.synthetic import make_problem


def _np(t):
    return None if t is None else t.numpy()


@pytest.mark.parametrize("parts", [2, 4])
def test_column_slices_concatenate_to_the_layer(parts):
    p = make_problem(5, 256, 128, 64, bias=True, seed=1)
    full = oracle.forward(p.x.numpy(), p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), p.bias.numpy(), 64)
    outs = [oracle.forward(p.x.numpy(), *(_np(t) for t in s), 64)
            for s in split_columns(p.qweight, p.qzeros, p.scales, p.bias, parts)]
    assert np.array_equal(np.concatenate(outs, axis=1), full)


@pytest.mark.parametrize("parts,g", [(2, 64), (4, 32), (2, -1)])
def test_row_slices_sum_to_the_layer(parts, g):
    p = make_problem(3, 256, 64, g, bias=True, seed=2)
    full = oracle.forward(p.x.numpy(), p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), p.bias.numpy(), g)
    x = p.x.numpy()
    acc = np.zeros_like(full)
    k0 = 0
    for (qw, qz, sc, gs) in split_rows(p.qweight, p.qzeros, p.scales, g, parts):
        kr = qw.shape[0]
        acc += oracle.forward(np.ascontiguousarray(x[:, k0:k0 + kr]), qw.numpy(), qz.numpy(), sc.numpy(), None, gs)
        k0 += kr
    acc += p.bias.numpy().astype(np.float64)
    assert np.allclose(acc, full, rtol=1e-12, atol=1e-12)


def test_concatenated_projections_equal_separate_ones():
    layers = [make_problem(4, 128, n, 32, bias=b, seed=n) for n, b in ((64, True), (32, False), (96, True))]
    x = layers[0].x.numpy()
    qw, qz, sc, b = concat_columns([(l.qweight, l.qzeros, l.scales, l.bias) for l in layers])
    fused = oracle.forward(x, qw.numpy(), qz.numpy(), sc.numpy(), b.numpy(), 32)
    sep = [oracle.forward(x, l.qweight.numpy(), l.qzeros.numpy(), l.scales.numpy(), _np(l.bias), 32) for l in layers]
    assert np.array_equal(fused, np.concatenate(sep, axis=1))


def test_split_rules():
    p = make_problem(1, 256, 64, 64, seed=3)
    with pytest.raises(ValueError):
        split_columns(p.qweight, p.qzeros, p.scales, None, 3)        # 64 / 3
    with pytest.raises(ValueError):
        split_columns(p.qweight, p.qzeros, p.scales, None, 16)       # 4-column slices
    with pytest.raises(ValueError):
        split_rows(p.qweight, p.qzeros, p.scales, 64, 8)             # 32 rows: half a group
    with pytest.raises(ValueError):
        split_rows(p.qweight, p.qzeros, p.scales, 64, 3)
    shards = split_rows(p.qweight, p.qzeros, p.scales, 64, 4)
    assert [s[0].shape[0] for s in shards] == [64] * 4 and all(s[3] == 64 for s in shards)


def test_column_parallel_forward_checks_shapes_before_any_launch():
    """Host-side argument checks of the gathered column-parallel forward: they
    raise before anything reaches the library (CPU tensors here)."""
    import torch
    from bit_weight_quantized_awq_gb300.shard import column_parallel_forward
    a = make_problem(1, 256, 64, 64, seed=3)
    b = make_problem(1, 128, 64, 64, seed=4)
    sa = (a.qweight, a.qzeros, a.scales, None)
    with pytest.raises(ValueError, match="no shards"):
        column_parallel_forward(a.x, [], 64)
    with pytest.raises(ValueError, match="in_features"):
        column_parallel_forward(a.x, [sa, (b.qweight, b.qzeros, b.scales, None)], 64)
    with pytest.raises(ValueError, match="features"):
        column_parallel_forward(b.x, [sa], 64)
    with pytest.raises(ValueError, match="CUDA"):
        column_parallel_forward(a.x, [sa], 64)
    with pytest.raises(ValueError):
        column_parallel_forward(a.x, [sa], 64, out=torch.empty((1, 32), dtype=torch.float16))

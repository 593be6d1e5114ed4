"""Act-order g_idx layers on the host: the library's row sort
(awq_gidx_sort, a host routine) and the identity the sorted forward relies
on, checked on the oracle.

Linear Layer Factory page, Description (the GPTQ tuple's g_idx): when every
group holds K / G rows, sorting the rows by group gives a grouped layer with
the same zero points and scales, and y = x[:, perm] . W[perm] is the g_idx
forward with its terms reordered.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_quantized_awq_gb300 import AWQError, Status, gidx_sort
from bit_weight_quantized_awq_gb300.build import build
from bit_weight_quantized_awq_gb300.synthetic import make_problem


@pytest.fixture(scope="module", autouse=True)
def lib():
    build(quiet=True)


def act_order(K, G, seed):
    rng = np.random.default_rng(seed)
    return (np.arange(K) // (K // G)).astype(np.int32)[rng.permutation(K)].copy()


@pytest.mark.parametrize("K,G", [(4096, 32), (1088, 17), (64, 1), (48, 48)])
def test_sort_is_the_stable_order_by_group(K, G):
    t = act_order(K, G, seed=K)
    perm = gidx_sort(torch.from_numpy(t), G).numpy()
    assert np.array_equal(perm, np.argsort(t, kind="stable"))
    assert np.array_equal(t[perm], np.arange(K) // (K // G))


def test_sort_refuses_tables_that_are_not_act_order():
    K, G = 256, 4
    t = act_order(K, G, seed=1)
    bad = t.copy()
    bad[3] = G                                   # outside [0, G)
    uneven = t.copy()
    uneven[np.flatnonzero(t == 0)[0]] = 1        # group 1 gets K/G + 1 rows
    for table, groups in [(bad, G), (uneven, G), (t, 3), (t, 0)]:
        with pytest.raises(AWQError) as e:
            gidx_sort(torch.from_numpy(table), groups)
        assert e.value.status == Status.ERR_INVALID_ARG


@pytest.mark.parametrize("M,K,N,G", [(3, 256, 64, 4), (5, 1024, 128, 8)])
def test_sorted_layer_equals_the_gidx_layer_on_the_oracle(M, K, N, G):
    p = make_problem(M, K, N, K // G, bias=True, seed=M + K)
    t = act_order(K, G, seed=7)
    perm = gidx_sort(torch.from_numpy(t), G).numpy()
    x, qw, qz, sc, b = p.x.numpy(), p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), p.bias.numpy()
    y_gidx = oracle.forward_gidx(x, qw, qz, sc, t, b)
    y_sorted = oracle.forward(np.ascontiguousarray(x[:, perm]), np.ascontiguousarray(qw[perm]), qz, sc, b, K // G)
    assert np.allclose(y_sorted, y_gidx, rtol=1e-12, atol=1e-12)
    # the sorted weights are the grouped dequant of the table's weights, row for row
    w_gidx = oracle.dequant_gidx(qw, qz, sc, t)
    w_sorted = oracle.dequant(np.ascontiguousarray(qw[perm]), qz, sc, K // G)
    assert np.array_equal(w_sorted, w_gidx[perm])

"""GPU parity: every path of the CUDA library against the CPU oracle on the
same seeded inputs.

* awq_dequant: bit-exact against the oracle's fp16 weights.
* awq_linear_forward: |y_gpu - y_ref| <= 1e-3 + 4e-3 |y_ref| element by
  element, every path that can take the shape plus the automatic choice.
  Small and medium shapes compare every output; the full-size workloads
  compare sampled rows (always 0 and M-1) and column blocks (start, middle,
  ragged end).
* metamorphic identities that must hold bit for bit on the GPU.

Workloads (Predibase Lorax "AWQ WQLinear" page gives the layer, not the
shapes; these are 7B- and 70B-class projection shapes): decode M in
{1, 4, 16}; prefill M in {512, 2048, 8192}; full-row grouping (group_size -1)
on a 3-D x; N = 8; a 70B-class M sweep. Inputs follow the synthetic recipe:
x ~ N(0, 1), codes uniform on 0..15, scales ~ U[1e-3, 1e-2], bias ~ 0.1 N(0, 1).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_quantized_awq_gb300 import (Path, awq_last_device_status, awq_path_supported,
                                            dequant, linear_forward)
from bit_weight_quantized_awq_gb300.synthetic import Problem, make_activations, make_problem

from parity import assert_close, check_problem, paths_for, run_path, sample_rows

pytestmark = pytest.mark.gpu

DECODE_SHAPES = [(4096, 4096), (4096, 12288), (4096, 22016), (11008, 4096)]
PREFILL_SHAPES = [(4096, 12288), (4096, 22016), (11008, 4096)]
SWEEP_SHAPES = [(8192, 10240), (8192, 57344), (28672, 8192)]
SWEEP_M = [1, 2, 4, 8, 16, 32, 64, 128, 512, 2048, 8192]


# --------------------------------------------------------------------------
# dequant: bit-exact
# --------------------------------------------------------------------------

@pytest.mark.parametrize("K,N,g", [(512, 512, 128), (4096, 4096, 128), (4096, 8, -1),
                                   (336, 104, 48), (48, 8, 16), (1, 8, 1), (11008, 4096, 128),
                                   (768, 800, 64), (64, 256, 32)])
def test_dequant_bit_exact(gpu, K, N, g):
    p = make_problem(1, K, N, g, seed=11)
    ref = oracle.dequant(p.qweight.numpy(), p.qzeros.numpy(), p.scales.numpy(), g)
    W = dequant(p.qweight.cuda(), p.qzeros.cuda(), p.scales.cuda(), g)
    torch.cuda.synchronize()
    got = W.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref), f"{(got != ref).sum()} weights differ"


def test_dequant_bit_exact_extreme_scales(gpu):
    """Negative, subnormal and overflowing scales: one rounding, IEEE rules."""
    K, N, g = 64, 512, 32
    p = make_problem(1, K, N, g, seed=12)
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 65536, size=(K // g, N), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7C00) == 0x7C00] &= 0xBBFF     # no inf/NaN scales
    sc = torch.from_numpy(bits.view(np.float16).copy())
    ref = oracle.dequant(p.qweight.numpy(), p.qzeros.numpy(), bits, g)
    W = dequant(p.qweight.cuda(), p.qzeros.cuda(), sc.cuda(), g)
    torch.cuda.synchronize()
    assert np.array_equal(W.cpu().numpy().view(np.uint16), ref)


# --------------------------------------------------------------------------
# forward: tiny, decode, edge and ragged shapes, every output compared
# --------------------------------------------------------------------------

def test_tiny_case(gpu):
    check_problem(make_problem(1, 512, 512, 128, bias=True, seed=0))


@pytest.mark.parametrize("K,N", DECODE_SHAPES)
@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_shapes(gpu, M, K, N):
    check_problem(make_problem(M, K, N, 128, bias=False, seed=0))


@pytest.mark.parametrize("M,K,N,g,bias", [
    (32, 4096, 4096, 128, False),   # four token tiles, split tiles
    (24, 2112, 1056, 96, True),     # padded tokens, groups that split a warp's rows
])
def test_decode_four_token_tiles(gpu, M, K, N, g, bias):
    check_problem(make_problem(M, K, N, g, bias=bias, seed=M + 50))


def test_decode_four_token_tiles_wide(gpu):
    # 512-column tiles with 32 tokens, sampled rows and column blocks
    check_problem(make_problem(32, 4096, 32768, 128, bias=True, seed=83), full=False)


def test_minimum_n_edge(gpu):
    check_problem(make_problem(1, 4096, 8, -1, bias=True, seed=0))


@pytest.mark.parametrize("M,K,N,g,bias", [
    (5, 1024, 800, 64, True),      # ragged column tile
    (3, 336, 104, 48, False),      # N % 32 != 0, odd group size
    (17, 768, 288, -1, True),      # four token tiles, 15 of them padding
    (33, 768, 288, -1, True),      # M just above the decode limit
    (2, 48, 8, 16, False),
    (1, 16, 8, 1, True),           # group size 1
    (7, 1088, 4128, 64, True),     # ragged tile in N and K not a multiple of 128
    (33, 512, 1024, 128, False),
    (130, 1024, 768, 128, True),
    (257, 2048, 1056, 128, False),
])
def test_ragged_and_edge_shapes(gpu, M, K, N, g, bias):
    check_problem(make_problem(M, K, N, g, bias=bias, seed=M))


# Decode on 512-column tiles (N a multiple of 512 and at least 32768): a
# ragged last k-stage (K % 128 == 64, the 512-column stage holds 128 rows),
# groups that split a warp's rows (g = 32, 64, 96), each token-tile class
# (M <= 8, 9..16, 17..32), with and without bias. The host plan query checks
# that each shape really takes 512-column tiles; the oracle is compared on
# every row and on column blocks at the start, the middle and the ragged end.
WIDE_TILE_CASES = [
    (1, 1088, 32768, 32, True),
    (8, 4160, 33280, 64, False),
    (9, 2112, 32768, 96, True),
    (16, 1088, 40960, 32, False),
    (17, 4160, 32768, 64, True),
    (32, 2112, 33280, 96, False),
    (3, 4096, 32768, 128, True),     # whole groups, K a multiple of the stage
]


@pytest.mark.parametrize("M,K,N,g,bias", WIDE_TILE_CASES)
def test_wide_tile_decode(gpu, M, K, N, g, bias):
    from bit_weight_quantized_awq_gb300 import awq_decode_tile_columns
    assert awq_decode_tile_columns(M, K, N, g) == 512
    check_problem(make_problem(M, K, N, g, bias=bias, seed=M + 100), paths=[Path.DECODE, Path.AUTO],
                  full=False)


# The same split-group and ragged-stage cases on 256-column tiles (N below
# 32768), every output compared.
@pytest.mark.parametrize("M,K,N,g,bias", [
    (1, 1088, 8192, 32, True),
    (9, 2112, 8704, 96, False),
    (16, 4160, 16384, 64, True),
    (3, 4096, 8192, 128, True),
    (12, 11008, 12288, 128, True),
])
def test_narrow_tile_decode(gpu, M, K, N, g, bias):
    from bit_weight_quantized_awq_gb300 import awq_decode_tile_columns
    assert awq_decode_tile_columns(M, K, N, g) == 256
    check_problem(make_problem(M, K, N, g, bias=bias, seed=M + 100), full=K * N <= 4160 * 16384)


# Prefill with fewer tiles than SMs: every tile's k-stages are split between
# CTAs ("stream-K"), which leave fp32 pieces that the sum kernel adds up. All
# outputs are compared, and repeated runs must agree bit for bit (the pieces
# are added in contributor order).
@pytest.mark.parametrize("M,K,N,g,bias", [
    (40, 4096, 1024, 128, True),
    (200, 2112, 800, 96, True),     # ragged tile in N, groups that split a stage
    (129, 1088, 4128, 64, False),   # two token tiles, ragged K and N
    (512, 2112, 2080, 64, True),    # 256-row tiles, 4-5 contributors per tile (whole ranges inside a tile)
    (300, 4224, 4128, 128, False),  # 256-row tiles, ragged M, 5-6 contributors per tile
])
def test_prefill_stream_k(gpu, M, K, N, g, bias):
    p = make_problem(M, K, N, g, bias=bias, seed=M + 7)
    check_problem(p, paths=[Path.PREFILL])
    pg = p.to("cuda")
    y0 = run_path(pg, Path.PREFILL)
    for _ in range(3):
        assert torch.equal(run_path(pg, Path.PREFILL).view(torch.int16), y0.view(torch.int16))


# A last, partial wave that fills most SMs runs whole: one tile per CTA, no
# pieces, no sum kernel (the tile width stays 256 columns; at 152 SMs this
# shape has 130 tiles of 10 k-stages, where splitting would cost more than
# the idle SMs). Groups of 64 split every 64-row stage in two.
def test_last_wave_whole(gpu):
    p = make_problem(384, 640, 16640, 64, bias=True, seed=384)
    check_problem(p, paths=[Path.PREFILL], full=False)
    pg = p.to("cuda")
    y0 = run_path(pg, Path.PREFILL)
    assert torch.equal(run_path(pg, Path.PREFILL).view(torch.int16), y0.view(torch.int16))


# x larger than the L2 share the tile order plans for, on the fused kernel
# and on the GEMM core; sampled rows and column blocks:
#  * K = 4096, N = 2560: 18 row blocks of 256 in bands of 16 (the share
#    holds 16 row blocks; the last band is 2 rows high) x 10 column blocks;
#  * K = 11008, N = 4096: the share holds only 5 row blocks, fewer than a
#    wave needs with 16 column blocks, so bands are 10 row blocks high (the
#    last one 8).
@pytest.mark.parametrize("path", [Path.PREFILL, Path.DEQUANT_GEMM])
@pytest.mark.parametrize("K,N", [(4096, 2560), (11008, 4096)])
def test_banded_tile_order(gpu, path, K, N):
    check_problem(make_problem(4608, K, N, 128, bias=True, seed=4608), paths=[path], full=False)


# --------------------------------------------------------------------------
# full-size workloads: sampled rows and column blocks
# --------------------------------------------------------------------------

@pytest.mark.parametrize("K,N", PREFILL_SHAPES)
@pytest.mark.parametrize("M,bias", [(512, True), (2048, False), (8192, True)])
def test_prefill_shapes(gpu, M, K, N, bias):
    check_problem(make_problem(M, K, N, 128, bias=bias, seed=0), full=False)


def test_prefill_bias_reverse_pass(gpu):
    """The second pass of the bias alternation: with bias at M = 2048."""
    check_problem(make_problem(2048, 4096, 12288, 128, bias=True, seed=1), full=False)


def test_full_row_grouping_3d_input(gpu):
    p = make_problem(8 * 256, 4096, 4096, -1, bias=True, seed=0, x_shape=(8, 256, 4096))
    pg = p.to("cuda")
    for path in paths_for(p.M, p.K, p.N, -1):
        y = run_path(pg, path)
        assert tuple(y.shape) == (8, 256, 4096)
    check_problem(p, full=False)


_weights_cache = {}


def _sweep_weights(K, N):
    if (K, N) not in _weights_cache:
        _weights_cache.clear()
        _weights_cache[(K, N)] = make_problem(1, K, N, 128, bias=False, seed=0)
    return _weights_cache[(K, N)]


@pytest.mark.parametrize("K,N", SWEEP_SHAPES)
@pytest.mark.parametrize("M", SWEEP_M)
def test_70b_sweep(gpu, K, N, M):
    w = _sweep_weights(K, N)
    p = Problem(make_activations(M, K, seed=M), w.qweight, w.qzeros, w.scales, None, 128)
    check_problem(p, full=False, max_rows=16)


# --------------------------------------------------------------------------
# metamorphic identities (bit-exact on the GPU)
# --------------------------------------------------------------------------

META_SHAPES = [(1, 512, 512, 128), (4, 4096, 4096, 128), (16, 4096, 1024, 64),
               (64, 1024, 1024, 128), (512, 1024, 2048, 128)]


def _all_paths(M, K, N, g):
    return [p for p in paths_for(M, K, N, g) if p != Path.AUTO]


@pytest.mark.parametrize("M,K,N,g", META_SHAPES)
def test_doubling_scales_doubles_output(gpu, M, K, N, g):
    p = make_problem(M, K, N, g, seed=21).to("cuda")
    p2 = Problem(p.x, p.qweight, p.qzeros, p.scales * 2, None, g)
    for path in _all_paths(M, K, N, g):
        y1 = run_path(p, path).float()
        y2 = run_path(p2, path).float()
        normal = y1.abs() >= 2.0 ** -13   # doubling is exact outside the fp16 subnormal range
        assert torch.equal(y2[normal], 2 * y1[normal]), path.name


@pytest.mark.parametrize("M,K,N,g", META_SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_q_equal_z_gives_bias(gpu, M, K, N, g, with_bias):
    p = make_problem(M, K, N, g, bias=with_bias, seed=22).to("cuda")
    qw = p.qzeros.repeat_interleave(g, dim=0).contiguous()
    for path in _all_paths(M, K, N, g):
        y = run_path(Problem(p.x, qw, p.qzeros, p.scales, p.bias, g), path)
        if with_bias:
            assert torch.equal(y, p.bias.expand(M, N)), path.name
        else:
            assert torch.count_nonzero(y) == 0, path.name


@pytest.mark.parametrize("M,K,N", [(4, 4096, 4096), (1, 512, 512), (256, 1024, 1024)])
def test_group_minus_one_equals_group_k(gpu, M, K, N):
    p = make_problem(M, K, N, -1, bias=True, seed=23).to("cuda")
    for path in _all_paths(M, K, N, K):
        a = run_path(p, path)
        b = run_path(Problem(p.x, p.qweight, p.qzeros, p.scales, p.bias, K), path)
        assert torch.equal(a, b), path.name


@pytest.mark.parametrize("M,K,N,g", [(4, 4096, 4096, 128), (300, 1024, 2048, 128)])
def test_column_permutation_within_blocks(gpu, M, K, N, g):
    """Permuting whole int32 columns inside aligned 128-column blocks (with
    the matching scales, zeros and bias) permutes y the same way, exactly."""
    p = make_problem(M, K, N, g, bias=True, seed=24)
    words = N // 8
    rng = np.random.default_rng(5)
    perm = np.concatenate([b * 16 + rng.permutation(16) for b in range(words // 16)])
    cperm = (perm[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
    pp = Problem(p.x, p.qweight[:, perm].contiguous(), p.qzeros[:, perm].contiguous(),
                 p.scales[:, cperm].contiguous(), p.bias[cperm].contiguous(), g).to("cuda")
    pg = p.to("cuda")
    for path in _all_paths(M, K, N, g):
        y = run_path(pg, path)
        yp = run_path(pp, path)
        assert torch.equal(yp, y[:, torch.from_numpy(cperm).cuda()]), path.name


# --------------------------------------------------------------------------
# canaries: nothing outside the output is written
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,N,g", [(1, 4096, 8, -1), (5, 1024, 800, 64), (16, 4096, 4096, 128),
                                     (130, 1024, 768, 128), (3, 336, 104, 48)])
def test_output_canaries(gpu, M, K, N, g):
    p = make_problem(M, K, N, g, bias=True, seed=25).to("cuda")
    pad = 64
    for path in _all_paths(M, K, N, g):
        buf = torch.full((M * N + 2 * pad,), 12345.0, dtype=torch.float16, device="cuda")
        out = buf[pad:pad + M * N]
        run_path(p, path, out=out)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == 12345.0) and torch.all(buf[-pad:] == 12345.0), path.name
    wbuf = torch.full((K * N + 2 * pad,), -7.0, dtype=torch.float16, device="cuda")
    dequant(p.qweight, p.qzeros, p.scales, g, out=wbuf[pad:pad + K * N])
    torch.cuda.synchronize()
    assert torch.all(wbuf[:pad] == -7.0) and torch.all(wbuf[-pad:] == -7.0)


def test_m_zero_writes_nothing(gpu):
    p = make_problem(1, 512, 512, 128, seed=26).to("cuda")
    x0 = p.x[:0]
    y = linear_forward(x0, p.qweight, p.qzeros, p.scales, None, 128)
    assert y.shape == (0, 512)


def test_device_status_clean_after_suite_calls(gpu):
    assert awq_last_device_status(torch.cuda.current_stream().cuda_stream) == 0


def test_library_cross_check_cublas(gpu):
    """Informative cross-check against a library routine: dequantised W fed to
    torch.matmul (cuBLAS, fp16 in / fp32 accumulate) agrees within the same
    tolerance with the oracle."""
    p = make_problem(16, 4096, 4096, 128, bias=True, seed=27)
    pg = p.to("cuda")
    W = dequant(pg.qweight, pg.qzeros, pg.scales, 128)
    y = (pg.x.float() @ W.float() + pg.bias.float()).half()
    from parity import oracle_reference
    assert_close(y.cpu().numpy(), oracle_reference(p), "cuBLAS on awq_dequant")


# --------------------------------------------------------------------------
# back-to-back calls on one stream: each layer's output is the next one's
# input, and a later layer writes the buffer an earlier one read. The decode
# kernel may start streaming weights before the previous kernel has finished
# (programmatic dependent launch); it must still see that kernel's output and
# must not overwrite what it reads. The chained result has to equal, bit for
# bit, the same calls with a device synchronisation after each.
# --------------------------------------------------------------------------

def _chain_matches_serialised(M, path, KN):
    K = N = KN
    layers = [make_problem(M, K, N, 128, bias=(i == 1), seed=40 + i).to(torch.device("cuda"))
              for i in range(4)]
    x0 = make_activations(M, K, seed=7).cuda()

    def run(sync: bool) -> list:
        a = x0.clone()
        b = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        bufs, outs = [a, b], []
        for i, L in enumerate(layers):
            src, dst = bufs[i % 2], bufs[(i + 1) % 2]
            linear_forward(src, L.qweight, L.qzeros, L.scales, L.bias, L.group_size, path=path, out=dst)
            if sync:
                torch.cuda.synchronize()
                outs.append(dst.clone())
        torch.cuda.synchronize()
        return outs if sync else [bufs[len(layers) % 2].clone()]

    serial = run(sync=True)
    chained = run(sync=False)
    assert torch.equal(chained[0].view(torch.int16), serial[-1].view(torch.int16))
    # the first layer of the serial run against the oracle (sampled rows for
    # the widest layers)
    p0 = layers[0]
    rows = sample_rows(M, 16) if KN > 8192 else None
    ref = oracle.forward(x0.cpu().numpy(), p0.qweight.cpu().numpy(), p0.qzeros.cpu().numpy(),
                         p0.scales.cpu().numpy(), None, p0.group_size, rows=rows)
    got = serial[0].cpu().numpy()
    assert_close(got if rows is None else got[rows], ref, "chained layer 0")
    assert awq_last_device_status(torch.cuda.current_stream().cuda_stream) == 0


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("path", [Path.DECODE, Path.AUTO])
@pytest.mark.parametrize("KN", [2048, 8192])
def test_chained_layers_match_serialised(gpu, M, path, KN):
    _chain_matches_serialised(M, path, KN)


# Dequantise-then-GEMM over several windows of one scratch buffer, three
# calls back to back on one stream (each window's dequant rewrites the buffer
# the previous window's GEMM read). Every output of the three calls must be
# the same bits, and must agree with the fused kernel's (the same fp16 W,
# fp32 sums in another order) far inside the forward tolerance: a window read
# while being rewritten would break both. The oracle checks sampled outputs
# of this path in test_70b_sweep.
def test_dequant_gemm_windows_in_order(gpu):
    M, K, N = 96, 8192, 57344          # four windows of fp16 weights
    w = _sweep_weights(K, N)
    x = make_activations(M, K, seed=3).cuda()
    qw, qz, sc = w.qweight.cuda(), w.qzeros.cuda(), w.scales.cuda()
    outs = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for _ in range(3)]
    torch.cuda.synchronize()
    for y in outs:
        linear_forward(x, qw, qz, sc, None, 128, path=Path.DEQUANT_GEMM, out=y)
    fused = linear_forward(x, qw, qz, sc, None, 128, path=Path.PREFILL)
    torch.cuda.synchronize()
    assert awq_last_device_status(torch.cuda.current_stream().cuda_stream) == 0
    for y in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))
    a, b = outs[0].double(), fused.double()
    assert torch.isfinite(a).all()
    assert ((a - b).abs() <= 1e-4 + 1e-3 * b.abs()).all()


# The same chain on the tensor-core paths, which are launched as programmatic
# dependents too: the fused kernel requests its first stages' packed weights
# before waiting for the previous kernel, x and everything it writes after;
# the stream-K sum kernel lets the next layer's kernel be scheduled early.
# M = 512 at K = N = 2048 splits every tile along k (sum kernel in the
# chain); M = 2560 at K = N = 4096 has a whole wave and a split last wave;
# K = N = 12288 (288 MiB of fp16 weights) takes two dequantise-then-GEMM
# windows.
@pytest.mark.parametrize("M,KN", [(512, 2048), (2560, 4096), (64, 12288)])
@pytest.mark.parametrize("path", [Path.PREFILL, Path.DEQUANT_GEMM])
def test_chained_prefill_layers_match_serialised(gpu, M, KN, path):
    _chain_matches_serialised(M, path, KN)

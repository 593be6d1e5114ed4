"""GPU parity of the step before the forward: awq_pack and awq_quantize_rtn
against the CPU oracle, bit for bit (integer results).

awq_pack is the inverse of the unpacking every forward kernel performs (the
packed int32 layout of the Predibase Lorax "AWQ WQLinear" page, I/O
Contract, in this library's nibble order); awq_quantize_rtn inverts the
group-wise dequantisation (Overview: group-wise scaling) with
q = clamp(round_half_even(W / s) + z, 0, 15). Shapes cover 7B-class
projection matrices, ragged word counts, group_size -1 and odd groups; values
cover ties, clamping, zero and infinite quotients, and the round trip through
awq_dequant.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_quantized_awq_gb300 import dequant, pack, quantize_rtn
from bit_weight_quantized_awq_gb300.synthetic import make_problem

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("R,C", [(4096, 4096), (11008, 512), (3, 8), (37, 104), (1, 22016)])
def test_pack_bit_exact(gpu, R, C):
    g = torch.Generator().manual_seed(R + C)
    codes = torch.randint(0, 256, (R, C), dtype=torch.uint8, generator=g)   # high bits ignored
    got = pack(codes.cuda()).cpu().numpy()
    assert np.array_equal(got, oracle.pack(codes.numpy()))


@pytest.mark.parametrize("K,N,g", [(4096, 4096, 128), (4096, 12288, 128), (336, 104, 48),
                                   (64, 8, -1), (1024, 800, 64), (48, 16, 16)])
def test_quantize_bit_exact(gpu, K, N, g):
    """Random fp16 W spread over the whole code range and beyond."""
    p = make_problem(1, K, N, g, seed=K + N)
    gen = torch.Generator().manual_seed(K * 3 + N)
    G = p.scales.shape[0]
    gsz = K if g == -1 else g
    s64 = p.scales.double().repeat_interleave(gsz, dim=0)
    W = (torch.randn((K, N), generator=gen, dtype=torch.float64) * 9.0 * s64).half()
    got = quantize_rtn(W.cuda(), p.scales.cuda(), p.qzeros.cuda(), g).cpu().numpy()
    ref = oracle.quantize_rtn(W.numpy(), p.scales.numpy(), p.qzeros.numpy(), g)
    assert np.array_equal(got, ref), f"{(got != ref).sum()} words differ"


def test_quantize_ties_clamps_and_special_quotients(gpu):
    """Quotients on halves, just off halves, far out of range, 0/0, x/0,
    subnormal and infinite W, with zero points 0, 8 and 15."""
    t = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.375, 3.625, 100.0, -100.0, 7.5, -8.5,
                  0.0, 6.5, -7.5, -6.5])
    N = 64
    W = np.zeros((3, N), dtype=np.float16)
    s = np.full((3, N), 0.25, dtype=np.float16)
    W[0, :16] = (t * 0.25).astype(np.float16)
    W[0, 16:32] = (-t * 0.25).astype(np.float16)
    s[1, :8] = 0.0
    W[1, :8] = np.array([0.0, 1.0, -1.0, 0.0, 6e-8, -6e-8, np.inf, -np.inf], dtype=np.float16)
    W[1, 8:16] = np.array([6e-8, 1e-7, -6e-8, 65504, -65504, np.inf, -np.inf, 0.0], dtype=np.float16)
    s[2, :] = np.float16(6e-8)                  # smallest subnormal scale
    W[2, :] = (np.arange(N) - 32).astype(np.float16) * np.float16(6e-8)
    for zval in (0, 8, 15):
        z = np.full((3, N), zval, dtype=np.uint8)
        qz = oracle.pack(z)
        ref = oracle.quantize_rtn(W, s, qz, 1)
        got = quantize_rtn(torch.from_numpy(W).cuda(), torch.from_numpy(s).cuda(),
                           torch.from_numpy(qz).cuda(), 1).cpu().numpy()
        assert np.array_equal(got, ref), zval


def test_quantize_exact_halves_and_their_neighbours_over_all_scale_exponents(gpu):
    """Every half-integer quotient h in [-64.5, 64.5] for 512 scales spread
    over all fp16 exponents (normal and subnormal), with W = h * s where that
    is an fp16 value, and W one fp16 step above and below it: the quotients
    the rounding decision is most sensitive to."""
    rng = np.random.default_rng(12)
    bits = rng.integers(1, 0x7C00, size=512).astype(np.uint16)    # positive finite, nonzero
    svals = bits.view(np.float16)
    halves = np.arange(-129, 130, 2) / 2.0                         # -64.5 .. 64.5
    rows = []
    for h in halves:
        w = (h * svals.astype(np.float64)).astype(np.float16)
        rows += [w, np.nextafter(w, np.float16(np.inf)), np.nextafter(w, np.float16(-np.inf))]
    W = np.stack(rows).astype(np.float16)                          # [3 * 259, 512]
    W[~np.isfinite(W)] = np.float16(0)
    K, N = W.shape
    s = np.tile(svals, (K, 1))
    for zval in (0, 8):
        qz = oracle.pack(np.full((K, N), zval, dtype=np.uint8))
        ref = oracle.quantize_rtn(W, s, qz, 1)
        got = quantize_rtn(torch.from_numpy(W).cuda(), torch.from_numpy(s).cuda(),
                           torch.from_numpy(qz).cuda(), 1).cpu().numpy()
        assert np.array_equal(got, ref), f"z={zval}: {(got != ref).sum()} words differ"


@pytest.mark.parametrize("K,N,g", [(4096, 22016, 128), (11008, 4096, 128), (256, 64, -1)])
def test_quantize_inverts_dequant(gpu, K, N, g):
    """awq_quantize_rtn(awq_dequant(q)) == q for the synthetic scales."""
    p = make_problem(1, K, N, g, seed=5).to("cuda")
    W = dequant(p.qweight, p.qzeros, p.scales, g)
    back = quantize_rtn(W, p.scales, p.qzeros, g)
    assert torch.equal(back, p.qweight)


def test_pack_matches_layout_read_by_the_forward(gpu):
    """Codes packed on the GPU dequantise to the codes' values: unpacking is
    done by the forward kernels' layout, checked against the oracle."""
    K, N, g = 512, 256, 128
    gen = torch.Generator().manual_seed(8)
    q = torch.randint(0, 16, (K, N), dtype=torch.uint8, generator=gen)
    z = torch.randint(0, 16, (K // g, N), dtype=torch.uint8, generator=gen)
    s = (torch.rand((K // g, N), generator=gen) * 9e-3 + 1e-3).half()
    qw, qz = pack(q.cuda()), pack(z.cuda())
    W = dequant(qw, qz, s.cuda(), g).cpu().numpy().view(np.uint16)
    ref = oracle.dequant(oracle.pack(q.numpy()), oracle.pack(z.numpy()), s.numpy(), g)
    assert np.array_equal(W, ref)

"""Host-only checks of the C ABI: the library builds and loads, exports every
function ``include/awq_gb300.h`` declares, and returns the documented status
for every invalid argument before any CUDA call (so these run without a GPU).

Shape rules: Predibase Lorax "AWQ WQLinear" page, Description, __init__
(w_bit 4, out_features % 8 == 0, group_size -1 -> in_features,
in_features % group_size == 0).
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import bit_weight_quantized_awq_gb300 as awq
from bit_weight_quantized_awq_gb300 import Path, Status
from bit_weight_quantized_awq_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "awq_gb300.h")

A = 0x10000      # 16-byte aligned fake device address: never dereferenced here
B = 0x20000


@pytest.fixture(scope="module")
def lib():
    build(quiet=True)
    return awq.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(awq_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(awq.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", awq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(awq_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for s in Status:
        text = awq.awq_status_string(s)
        assert text.startswith("AWQ_"), text
    assert "unknown" in awq.awq_status_string(99)


def fwd(M=4, K=256, N=64, g=128, x=A, qw=A, qz=A, sc=A, bias=None, y=B, path=Path.AUTO):
    return awq.awq_linear_forward_path(x, qw, qz, sc, bias, y, M, K, N, g, None, path)


@pytest.mark.parametrize("kw", [
    dict(N=12), dict(N=0), dict(N=-8), dict(K=0), dict(K=-1), dict(g=0), dict(g=-2),
    dict(g=100), dict(K=256, g=512), dict(M=-1),
    dict(x=None), dict(qw=None), dict(qz=None), dict(sc=None), dict(y=None),
])
def test_forward_invalid_args(lib, kw):
    assert fwd(**kw) == Status.ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(x=A + 2), dict(qw=A + 4), dict(qz=A + 8), dict(sc=A + 2),
                                dict(y=B + 2), dict(bias=A + 6)])
def test_forward_misaligned(lib, kw):
    assert fwd(**kw) == Status.ERR_MISALIGNED


def test_forward_m_zero_is_noop(lib):
    assert fwd(M=0) == Status.OK
    assert fwd(M=0, g=-1) == Status.OK
    assert awq.awq_linear_forward(A, A, A, A, None, B, 0, 4096, 8, -1, None) == Status.OK


def test_forward_bad_path(lib):
    assert fwd(path=7) == Status.ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(N=12), dict(g=0), dict(g=-3), dict(K=256, g=96)])
def test_dequant_invalid(lib, kw):
    K, N, g = kw.get("K", 256), kw.get("N", 64), kw.get("g", 128)
    assert awq.awq_dequant(A, A, A, B, K, N, g, None) == Status.ERR_INVALID_ARG


def test_dequant_null_and_misaligned(lib):
    assert awq.awq_dequant(None, A, A, B, 256, 64, 128, None) == Status.ERR_INVALID_ARG
    assert awq.awq_dequant(A, A, A, None, 256, 64, 128, None) == Status.ERR_INVALID_ARG
    assert awq.awq_dequant(A + 4, A, A, B, 256, 64, 128, None) == Status.ERR_MISALIGNED
    assert awq.awq_dequant(A, A, A, B + 8, 256, 64, 128, None) == Status.ERR_MISALIGNED


def test_pack_argument_rules(lib):
    assert awq.awq_pack(A, B, 4, 12, None) == Status.ERR_INVALID_ARG     # cols % 8
    assert awq.awq_pack(A, B, 4, 0, None) == Status.ERR_INVALID_ARG
    assert awq.awq_pack(A, B, -1, 8, None) == Status.ERR_INVALID_ARG
    assert awq.awq_pack(None, B, 4, 8, None) == Status.ERR_INVALID_ARG
    assert awq.awq_pack(A + 8, B, 4, 8, None) == Status.ERR_MISALIGNED
    assert awq.awq_pack(A, B + 4, 4, 8, None) == Status.ERR_MISALIGNED
    assert awq.awq_pack(None, None, 0, 8, None) == Status.OK            # nothing to do


@pytest.mark.parametrize("kw", [dict(N=12), dict(g=0), dict(g=-3), dict(K=256, g=96), dict(K=0)])
def test_quantize_invalid(lib, kw):
    K, N, g = kw.get("K", 256), kw.get("N", 64), kw.get("g", 128)
    assert awq.awq_quantize_rtn(A, A, A, B, K, N, g, None) == Status.ERR_INVALID_ARG


def test_quantize_null_and_misaligned(lib):
    assert awq.awq_quantize_rtn(None, A, A, B, 256, 64, 128, None) == Status.ERR_INVALID_ARG
    assert awq.awq_quantize_rtn(A, A, A, None, 256, 64, 128, None) == Status.ERR_INVALID_ARG
    assert awq.awq_quantize_rtn(A + 2, A, A, B, 256, 64, 128, None) == Status.ERR_MISALIGNED
    assert awq.awq_quantize_rtn(A, A, A + 4, B, 256, 64, 128, None) == Status.ERR_MISALIGNED


def test_gidx_argument_rules(lib):
    dq = lambda **k: awq.awq_dequant_gidx(k.get("qw", A), A, A, k.get("gi", A), k.get("W", B),
                                          k.get("K", 256), k.get("N", 64), k.get("G", 4), None)
    assert dq(N=12) == Status.ERR_INVALID_ARG
    assert dq(G=0) == Status.ERR_INVALID_ARG
    assert dq(K=0) == Status.ERR_INVALID_ARG
    assert dq(gi=None) == Status.ERR_INVALID_ARG
    assert dq(gi=A + 4) == Status.ERR_MISALIGNED
    assert dq(W=B + 2) == Status.ERR_MISALIGNED
    fw = lambda **k: awq.awq_linear_forward_gidx(k.get("x", A), A, A, A, k.get("gi", A), None, B,
                                                 k.get("M", 4), k.get("K", 256), k.get("N", 64),
                                                 k.get("G", 4), None)
    assert fw(N=40) == Status.ERR_INVALID_ARG      # N % 32 for the tensor-core core
    assert fw(K=72) == Status.ERR_INVALID_ARG      # K % 16
    assert fw(G=-1) == Status.ERR_INVALID_ARG
    assert fw(M=-1) == Status.ERR_INVALID_ARG
    assert fw(gi=None) == Status.ERR_INVALID_ARG
    assert fw(x=A + 2) == Status.ERR_MISALIGNED
    assert fw(M=0) == Status.OK


def test_row_piece_argument_rules(lib):
    rows = lambda **k: awq.awq_linear_forward_rows(k.get("x", A), k.get("ldx", 256), A, A, A, k.get("y32", B),
                                                   k.get("M", 4), k.get("K", 256), k.get("N", 64),
                                                   k.get("g", 128), None)
    assert rows(ldx=128) == Status.ERR_INVALID_ARG     # ldx < K
    assert rows(ldx=260) == Status.ERR_INVALID_ARG     # ldx % 8
    assert rows(N=12) == Status.ERR_INVALID_ARG
    assert rows(M=-1) == Status.ERR_INVALID_ARG
    assert rows(y32=None) == Status.ERR_INVALID_ARG
    assert rows(x=A + 2) == Status.ERR_MISALIGNED
    assert rows(y32=B + 4) == Status.ERR_MISALIGNED
    assert rows(M=0, x=None, y32=None) == Status.OK
    assert awq.awq_finish_rows(A, None, B, 4, 12, None) == Status.ERR_INVALID_ARG
    assert awq.awq_finish_rows(None, None, B, 4, 64, None) == Status.ERR_INVALID_ARG
    assert awq.awq_finish_rows(A, A + 2, B, 4, 64, None) == Status.ERR_MISALIGNED
    assert awq.awq_finish_rows(None, None, None, 0, 64, None) == Status.OK


def test_path_support_rules(lib):
    # the generic kernel takes every valid shape, nothing takes an invalid one
    for (M, K, N, g) in [(1, 4096, 8, -1), (3, 48, 104, 16), (5, 336, 800, 48), (1, 1, 8, 1)]:
        assert awq.awq_path_supported(M, K, N, g, Path.GENERIC) == 1
        assert awq.awq_select_path(M, K, N, g) in (Path.GENERIC, Path.DECODE, Path.PREFILL,
                                                   Path.DEQUANT_GEMM)
    assert awq.awq_path_supported(1, 4096, 12, 128, Path.GENERIC) == 0
    assert awq.awq_select_path(1, 4096, 12, 128) == -1
    assert awq.awq_select_path(-1, 4096, 4096, 128) == -1
    # a forced path that cannot take the shape is refused before any launch
    for path in (Path.DECODE, Path.PREFILL, Path.DEQUANT_GEMM):
        if not awq.awq_path_supported(1, 4096, 8, -1, path):
            assert fwd(M=1, K=4096, N=8, g=-1, path=path) == Status.ERR_INVALID_ARG


def test_automatic_path_follows_the_measured_crossovers(lib):
    # decode through 32 tokens, the fused tcgen05 kernel up to 6143, then the
    # weights dequantised once and the plain tcgen05 GEMM (when K <= 16384)
    for M, want in [(1, Path.DECODE), (32, Path.DECODE), (33, Path.PREFILL), (2048, Path.PREFILL),
                    (6143, Path.PREFILL), (6144, Path.DEQUANT_GEMM), (8192, Path.DEQUANT_GEMM)]:
        assert awq.awq_select_path(M, 4096, 12288, 128) == want, M
    assert awq.awq_select_path(8192, 16384, 8192, 128) == Path.DEQUANT_GEMM
    assert awq.awq_select_path(8192, 28672, 8192, 128) == Path.PREFILL
    for path in (Path.PREFILL, Path.DEQUANT_GEMM):
        assert awq.awq_path_supported(2048, 4096, 12288, 128, path) == 1
        assert awq.awq_path_supported(2048, 4100, 12288, -1, path) == 0      # K % 16


def test_launch_count_rules_without_a_device(lib):
    # answers that need no SM count: invalid shapes, M = 0, one-kernel paths
    assert awq.awq_forward_launches(1, 4096, 12, 128, Path.AUTO) == -1
    assert awq.awq_forward_launches(-1, 4096, 4096, 128, Path.AUTO) == -1
    assert awq.awq_forward_launches(0, 4096, 4096, 128, Path.PREFILL) == 0
    assert awq.awq_forward_launches(1, 4096, 4096, 128, Path.AUTO) == 1        # decode
    assert awq.awq_forward_launches(7, 4096, 4096, 128, Path.GENERIC) == 1
    assert awq.awq_forward_launches(1, 4096, 8, -1, Path.PREFILL) == -1       # path cannot serve it


def test_layer_checks_on_host():
    qw = torch.zeros((256, 8), dtype=torch.int32)
    qz = torch.zeros((2, 8), dtype=torch.int32)
    sc = torch.zeros((2, 64), dtype=torch.float16)
    layer = awq.AWQLinear(4, 128, qw, qz, sc, None)
    assert layer.in_features == 256 and layer.out_features == 64 and layer.weight is qw
    assert awq.AWQLinear(4, -1, qw, qz[:1], sc[:1], None).group_size == 256
    with pytest.raises(ValueError):
        awq.AWQLinear(8, 128, qw, qz, sc, None)
    with pytest.raises(ValueError):
        awq.AWQLinear(4, 100, qw, qz, sc, None)
    with pytest.raises(ValueError):
        awq.AWQLinear(4, 128, qw, qz[:1], sc, None)
    with pytest.raises(ValueError):
        awq.AWQLinear(4, 128, qw, qz, sc, torch.zeros(63, dtype=torch.float16))
    # no CPU fallback: CPU tensors are refused loudly
    with pytest.raises(ValueError):
        layer(torch.zeros((1, 256), dtype=torch.float16))


def test_missing_library_fails_loudly(tmp_path):
    code = ("import bit_weight_quantized_awq_gb300._binding as b\n"
            f"b.load_library({str(tmp_path / 'nope.so')!r})\n")
    r = subprocess.run(["python", "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode != 0 and "not found" in r.stderr


def test_decode_tile_columns_plan(lib):
    """Host-only plan query: 512-column decode tiles exactly when N is a
    multiple of 512 and at least 32768; 0 where the decode kernel does not
    serve the shape; -1 for an invalid shape."""
    q = awq.awq_decode_tile_columns
    assert q(1, 4096, 32768, 128) == 512
    assert q(32, 2112, 33280, 96) == 512
    assert q(1, 4096, 32256, 128) == 256      # a multiple of 512, below 32768
    assert q(1, 4096, 33024, 128) == 256      # at least 32768, not a multiple of 512
    assert q(16, 4096, 22016, 128) == 256
    assert q(33, 4096, 4096, 128) == 0        # more rows than the decode kernel takes
    assert q(1, 4096, 8, -1) == 0             # N below one 32-column TMA row
    assert q(1, 4096, 12, 128) == -1          # N % 8 != 0


def test_fault_test_build_exports_the_switch_and_the_main_library_does_not(lib):
    """The timeout switch exists only in the fault-test build, which the GPU
    timeout tests load; the library users link has no such symbol."""
    from bit_weight_quantized_awq_gb300.build import FAULT_LIB
    main = subprocess.run(["nm", "-D", "--defined-only", awq.LIB_PATH], capture_output=True,
                          text=True, check=True).stdout
    ft = subprocess.run(["nm", "-D", "--defined-only", FAULT_LIB], capture_output=True,
                        text=True, check=True).stdout
    assert "awq_test_inject_fault" not in main
    assert re.search(r"\sT\sawq_test_inject_fault\b", ft)
    for n in awq.EXPORTED:
        assert re.search(rf"\sT\s{n}\b", ft), n


@pytest.mark.parametrize("args", [(-1, 4096, 4096, 0), (1, 0, 4096, 0), (1, 4096, 0, 0), (1, 4096, 4096, 4),
                                  (1, 4096, 4096, 0xFFFFFFFF)])
def test_reserve_invalid_args(lib, args):
    """awq_reserve checks its bounds and flags before any CUDA call."""
    assert awq.awq_reserve(*args, None) == Status.ERR_INVALID_ARG

"""ctypes front end of the plain-C oracle (``awq_oracle.c``).

TEST INFRASTRUCTURE: see the package docstring for who may import this.

Arrays are numpy. fp16 tensors are passed as their uint16 bit patterns (a
``np.float16`` array is accepted and viewed as ``np.uint16``); qweight and
qzeros are int32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "awq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ``awq_oracle.c`` with gcc into ``oracle/_build/liboracle.so``.

    ``-ffp-contract=off`` keeps a * b + c as two roundings on every host, so
    the fp64 sums are the same on x86-64 and aarch64.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # A test that plants a mistake in a copy of the oracle points this
        # variable at the copy's library; nothing else sets it.
        override = os.environ.get("AWQ_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        lib.awq_oracle_f16_to_f64.restype = ctypes.c_double
        lib.awq_oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.awq_oracle_f64_to_f16.restype = ctypes.c_uint16
        lib.awq_oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.awq_oracle_f64_to_f16_array.restype = None
        lib.awq_oracle_f64_to_f16_array.argtypes = [_P, _I64, _P]
        lib.awq_oracle_f16_to_f64_array.restype = None
        lib.awq_oracle_f16_to_f64_array.argtypes = [_P, _I64, _P]
        lib.awq_oracle_resolve_group.restype = ctypes.c_int
        lib.awq_oracle_resolve_group.argtypes = [_I64, _I64, _I64, ctypes.POINTER(_I64)]
        lib.awq_oracle_unpack.restype = ctypes.c_int
        lib.awq_oracle_unpack.argtypes = [_P, _I64, _I64, _P]
        lib.awq_oracle_dequant.restype = ctypes.c_int
        lib.awq_oracle_dequant.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P]
        lib.awq_oracle_dequant_gidx.restype = ctypes.c_int
        lib.awq_oracle_dequant_gidx.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P]
        lib.awq_oracle_forward_gidx.restype = ctypes.c_int
        lib.awq_oracle_forward_gidx.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                                _P, _I64, ctypes.c_int, _P]
        lib.awq_oracle_pack.restype = ctypes.c_int
        lib.awq_oracle_pack.argtypes = [_P, _I64, _I64, _P]
        lib.awq_oracle_quantize_rtn.restype = ctypes.c_int
        lib.awq_oracle_quantize_rtn.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P]
        lib.awq_oracle_forward.restype = ctypes.c_int
        lib.awq_oracle_forward.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                           _P, _I64, ctypes.c_int, _P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected fp16 bits (uint16 or float16), got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    if a.dtype != np.int32:
        raise TypeError(f"expected int32, got {a.dtype}")
    return a


def f64_to_f16_bits(v) -> np.ndarray:
    """Round doubles to binary16 (nearest, ties to even); returns uint16 bits."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().awq_oracle_f64_to_f16_array(_ptr(v), v.size, _ptr(out))
    return out


def f16_bits_to_f64(h) -> np.ndarray:
    """Exact value of binary16 bit patterns as doubles."""
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float64)
    _load().awq_oracle_f16_to_f64_array(_ptr(h), h.size, _ptr(out))
    return out


def resolve_group(in_features: int, out_features: int, group_size: int) -> int | None:
    """group_size after the -1 rule, or None if the shape is rejected."""
    g = _I64(0)
    rc = _load().awq_oracle_resolve_group(in_features, out_features, group_size, ctypes.byref(g))
    return None if rc else g.value


def unpack(packed, out_features: int | None = None) -> np.ndarray:
    """int32 [R, N/8] -> uint8 codes [R, N]."""
    packed = _i32(packed)
    rows, words = packed.shape
    n = 8 * words if out_features is None else out_features
    out = np.empty((rows, n), dtype=np.uint8)
    rc = _load().awq_oracle_unpack(_ptr(packed), rows, n, _ptr(out))
    if rc:
        raise ValueError("oracle rejected the unpack shape")
    return out


def pack(codes) -> np.ndarray:
    """uint8 codes [R, C] (low 4 bits used) -> int32 [R, C/8]; column 8j + i of
    a row goes to nibble i of word j."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    out = np.empty((rows, cols // 8), dtype=np.int32)
    rc = _load().awq_oracle_pack(_ptr(codes), rows, cols, _ptr(out))
    if rc:
        raise ValueError("oracle rejected the pack shape")
    return out


def quantize_rtn(W, scales, qzeros, group_size: int) -> np.ndarray:
    """Round-to-nearest codes of fp16 W [K, N] with the given fp16 scales
    [G, N] and packed zero points [G, N/8], packed: int32 [K, N/8].

    q = clamp(round_half_even(W / s) + z, 0, 15); a NaN quotient counts as 0.
    """
    W, scales, qzeros = _u16(W), _u16(scales), _i32(qzeros)
    K, N = W.shape
    g = resolve_group(K, N, group_size)
    if g is None:
        raise ValueError("oracle rejected the shape")
    if qzeros.shape != (K // g, N // 8) or scales.shape != (K // g, N):
        raise ValueError("qzeros/scales shape does not match W and group_size")
    out = np.empty((K, N // 8), dtype=np.int32)
    rc = _load().awq_oracle_quantize_rtn(_ptr(W), _ptr(scales), _ptr(qzeros), K, N, group_size,
                                         _ptr(out))
    if rc:
        raise RuntimeError(f"oracle quantize failed ({rc})")
    return out


def dequant(qweight, qzeros, scales, group_size: int) -> np.ndarray:
    """W16 bit patterns [K, N] (uint16)."""
    qweight, qzeros, scales = _i32(qweight), _i32(qzeros), _u16(scales)
    K, words = qweight.shape
    N = 8 * words
    g = resolve_group(K, N, group_size)
    if g is None:
        raise ValueError("oracle rejected the shape")
    if qzeros.shape != (K // g, words) or scales.shape != (K // g, N):
        raise ValueError("qzeros/scales shape does not match qweight and group_size")
    out = np.empty((K, N), dtype=np.uint16)
    rc = _load().awq_oracle_dequant(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N,
                                    group_size, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle dequant failed ({rc})")
    return out


def forward(x, qweight, qzeros, scales, bias, group_size: int, rows=None,
            threads: int | None = None) -> np.ndarray:
    """fp64 y [len(rows), N] (all rows of x when ``rows`` is None).

    ``x`` is fp16 [M, K]; a higher-rank x is flattened to 2-D first, which is
    forward step 1 on the WQLinear page. The result keeps the 2-D shape.
    """
    x = _u16(x)
    x = x.reshape(-1, x.shape[-1])
    qweight, qzeros, scales = _i32(qweight), _i32(qzeros), _u16(scales)
    bias = None if bias is None else _u16(bias)
    M, K = x.shape
    if qweight.shape[0] != K:
        raise ValueError("x and qweight disagree on in_features")
    N = 8 * qweight.shape[1]
    g = resolve_group(K, N, group_size)
    if g is None:
        raise ValueError("oracle rejected the shape")
    if qzeros.shape != (K // g, N // 8) or scales.shape != (K // g, N):
        raise ValueError("qzeros/scales shape does not match qweight and group_size")
    if bias is not None and bias.shape != (N,):
        raise ValueError("bias must have shape [N]")
    if rows is None:
        rows_a = np.arange(M, dtype=np.int64)
    else:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64)
    if threads is None:
        threads = os.cpu_count() or 1
    y = np.empty((rows_a.size, N), dtype=np.float64)
    rc = _load().awq_oracle_forward(_ptr(x), _ptr(qweight), _ptr(qzeros), _ptr(scales),
                                    _ptr(bias), M, K, N, group_size, _ptr(rows_a),
                                    rows_a.size, int(threads), _ptr(y))
    if rc:
        raise RuntimeError(f"oracle forward failed ({rc})")
    return y


def _gidx(g_idx, K):
    g_idx = np.ascontiguousarray(g_idx, dtype=np.int32)
    if g_idx.shape != (K,):
        raise ValueError("g_idx must have shape [K]")
    return g_idx


def dequant_gidx(qweight, qzeros, scales, g_idx) -> np.ndarray:
    """W16 bit patterns [K, N] with the group of row k taken from g_idx[k]."""
    qweight, qzeros, scales = _i32(qweight), _i32(qzeros), _u16(scales)
    K, words = qweight.shape
    N = 8 * words
    G = scales.shape[0]
    g_idx = _gidx(g_idx, K)
    if qzeros.shape != (G, words) or scales.shape != (G, N):
        raise ValueError("qzeros/scales shape does not match qweight")
    out = np.empty((K, N), dtype=np.uint16)
    rc = _load().awq_oracle_dequant_gidx(_ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx),
                                         K, N, G, _ptr(out))
    if rc:
        raise ValueError(f"oracle rejected the g_idx problem ({rc})")
    return out


def forward_gidx(x, qweight, qzeros, scales, g_idx, bias, rows=None,
                 threads: int | None = None) -> np.ndarray:
    """fp64 y with the group of input row k taken from g_idx[k]."""
    x = _u16(x)
    x = x.reshape(-1, x.shape[-1])
    qweight, qzeros, scales = _i32(qweight), _i32(qzeros), _u16(scales)
    bias = None if bias is None else _u16(bias)
    M, K = x.shape
    N = 8 * qweight.shape[1]
    G = scales.shape[0]
    g_idx = _gidx(g_idx, K)
    if qweight.shape[0] != K or qzeros.shape != (G, N // 8) or scales.shape != (G, N):
        raise ValueError("shapes do not match")
    rows_a = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    if threads is None:
        threads = os.cpu_count() or 1
    y = np.empty((rows_a.size, N), dtype=np.float64)
    rc = _load().awq_oracle_forward_gidx(_ptr(x), _ptr(qweight), _ptr(qzeros), _ptr(scales),
                                         _ptr(g_idx), _ptr(bias), M, K, N, G, _ptr(rows_a),
                                         rows_a.size, int(threads), _ptr(y))
    if rc:
        raise RuntimeError(f"oracle forward_gidx failed ({rc})")
    return y

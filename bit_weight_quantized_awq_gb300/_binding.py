"""ctypes binding of ``include/awq_gb300.h``: the same entry points, the same
names and arguments, pointers and streams passed as integers. Argument
marshalling only; every step of the computation runs in the CUDA library.

The library is built in-tree (``_build/libawq_gb300.so``). Loading fails
loudly if it is missing: there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libawq_gb300.so")

# Every function the header declares; tests check the library exports them.
EXPORTED = (
    "awq_linear_forward",
    "awq_linear_forward_path",
    "awq_path_supported",
    "awq_select_path",
    "awq_forward_launches",
    "awq_decode_tile_columns",
    "awq_dequant",
    "awq_status_string",
    "awq_last_device_status",
    "awq_shutdown",
    "awq_linear_forward_decode_noalloc",
    "awq_gemm_f16",
    "awq_pack",
    "awq_quantize_rtn",
    "awq_dequant_gidx",
    "awq_linear_forward_gidx",
    "awq_linear_forward_rows",
    "awq_finish_rows",
    "awq_gidx_sort",
    "awq_permute_rows",
    "awq_linear_forward_sorted",
    "awq_reserve",
)

RESERVE_SORTED = 1
RESERVE_GIDX = 2


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_ARG = 1
    ERR_MISALIGNED = 2
    ERR_CUDA = 3
    ERR_TIMEOUT = 4
    ERR_TOO_LARGE = 5


class Path(enum.IntEnum):
    AUTO = 0
    GENERIC = 1
    DECODE = 2
    PREFILL = 3
    DEQUANT_GEMM = 4


class AWQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        super().__init__(f"{where}: {awq_status_string(status)}")


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads the CUDA library once. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"AWQ CUDA library not found at {p}; build it with "
                "`python -m bit_weight_quantized_awq_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(p)
        fwd_args = [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]
        lib.awq_linear_forward.argtypes = fwd_args
        lib.awq_linear_forward.restype = _INT
        lib.awq_linear_forward_path.argtypes = fwd_args + [_INT]
        lib.awq_linear_forward_path.restype = _INT
        lib.awq_path_supported.argtypes = [_I64, _I64, _I64, _I64, _INT]
        lib.awq_path_supported.restype = _INT
        lib.awq_select_path.argtypes = [_I64, _I64, _I64, _I64]
        lib.awq_select_path.restype = _INT
        lib.awq_forward_launches.argtypes = [_I64, _I64, _I64, _I64, _INT]
        lib.awq_forward_launches.restype = _INT
        lib.awq_decode_tile_columns.argtypes = [_I64, _I64, _I64, _I64]
        lib.awq_decode_tile_columns.restype = _INT
        lib.awq_dequant.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P]
        lib.awq_dequant.restype = _INT
        lib.awq_status_string.argtypes = [_INT]
        lib.awq_status_string.restype = ctypes.c_char_p
        lib.awq_last_device_status.argtypes = [_P]
        lib.awq_last_device_status.restype = _INT
        lib.awq_linear_forward_decode_noalloc.argtypes = fwd_args
        lib.awq_linear_forward_decode_noalloc.restype = _INT
        lib.awq_gemm_f16.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P]
        lib.awq_gemm_f16.restype = _INT
        lib.awq_dequant_gidx.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]
        lib.awq_dequant_gidx.restype = _INT
        lib.awq_linear_forward_gidx.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]
        lib.awq_linear_forward_gidx.restype = _INT
        lib.awq_linear_forward_rows.argtypes = [_P, _I64, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]
        lib.awq_linear_forward_rows.restype = _INT
        lib.awq_gidx_sort.argtypes = [_P, _I64, _I64, _P]
        lib.awq_gidx_sort.restype = _INT
        lib.awq_permute_rows.argtypes = [_P, _P, _P, _I64, _I64, _P]
        lib.awq_permute_rows.restype = _INT
        lib.awq_linear_forward_sorted.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]
        lib.awq_linear_forward_sorted.restype = _INT
        lib.awq_finish_rows.argtypes = [_P, _P, _P, _I64, _I64, _P]
        lib.awq_finish_rows.restype = _INT
        lib.awq_pack.argtypes = [_P, _P, _I64, _I64, _P]
        lib.awq_pack.restype = _INT
        lib.awq_quantize_rtn.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P]
        lib.awq_quantize_rtn.restype = _INT
        lib.awq_reserve.argtypes = [_I64, _I64, _I64, ctypes.c_uint, _P]
        lib.awq_reserve.restype = _INT
        lib.awq_shutdown.argtypes = []
        lib.awq_shutdown.restype = None
        _lib = lib
        return lib


# ---- the C entry points, one to one ----

def awq_linear_forward(x, qweight, qzeros, scales, bias, y, M, K, N, group_size, stream) -> int:
    return load_library().awq_linear_forward(x, qweight, qzeros, scales, bias, y,
                                             M, K, N, group_size, stream)


def awq_linear_forward_path(x, qweight, qzeros, scales, bias, y, M, K, N, group_size, stream,
                            path) -> int:
    return load_library().awq_linear_forward_path(x, qweight, qzeros, scales, bias, y,
                                                  M, K, N, group_size, stream, int(path))


def awq_path_supported(M, K, N, group_size, path) -> int:
    return load_library().awq_path_supported(M, K, N, group_size, int(path))


def awq_select_path(M, K, N, group_size) -> int:
    return load_library().awq_select_path(M, K, N, group_size)


def awq_forward_launches(M, K, N, group_size, path=0) -> int:
    return load_library().awq_forward_launches(M, K, N, group_size, int(path))


def awq_decode_tile_columns(M, K, N, group_size) -> int:
    return load_library().awq_decode_tile_columns(M, K, N, group_size)


def awq_dequant(qweight, qzeros, scales, W, K, N, group_size, stream) -> int:
    return load_library().awq_dequant(qweight, qzeros, scales, W, K, N, group_size, stream)


def awq_gemm_f16(x, W, bias, y, M, K, N, stream) -> int:
    return load_library().awq_gemm_f16(x, W, bias, y, M, K, N, stream)


def awq_dequant_gidx(qweight, qzeros, scales, g_idx, W, K, N, G, stream) -> int:
    return load_library().awq_dequant_gidx(qweight, qzeros, scales, g_idx, W, K, N, G, stream)


def awq_linear_forward_gidx(x, qweight, qzeros, scales, g_idx, bias, y, M, K, N, G, stream) -> int:
    return load_library().awq_linear_forward_gidx(x, qweight, qzeros, scales, g_idx, bias, y,
                                                  M, K, N, G, stream)


def awq_gidx_sort(g_idx, K, G, perm) -> int:
    return load_library().awq_gidx_sort(g_idx, K, G, perm)


def awq_permute_rows(qweight, perm, qweight_sorted, K, N, stream) -> int:
    return load_library().awq_permute_rows(qweight, perm, qweight_sorted, K, N, stream)


def awq_linear_forward_sorted(x, perm, qweight_sorted, qzeros, scales, bias, y, M, K, N, group_size,
                              stream) -> int:
    return load_library().awq_linear_forward_sorted(x, perm, qweight_sorted, qzeros, scales, bias, y,
                                                    M, K, N, group_size, stream)


def awq_linear_forward_rows(x, ldx, qweight, qzeros, scales, y32, M, K, N, group_size, stream) -> int:
    return load_library().awq_linear_forward_rows(x, ldx, qweight, qzeros, scales, y32, M, K, N,
                                                  group_size, stream)


def awq_finish_rows(y32, bias, y, M, N, stream) -> int:
    return load_library().awq_finish_rows(y32, bias, y, M, N, stream)


def awq_pack(codes, packed, rows, cols, stream) -> int:
    return load_library().awq_pack(codes, packed, rows, cols, stream)


def awq_quantize_rtn(W, scales, qzeros, qweight, K, N, group_size, stream) -> int:
    return load_library().awq_quantize_rtn(W, scales, qzeros, qweight, K, N, group_size, stream)


def awq_status_string(status) -> str:
    return load_library().awq_status_string(int(status)).decode()


def awq_last_device_status(stream) -> int:
    return load_library().awq_last_device_status(stream)


def awq_reserve(max_M, max_K, max_N, flags, stream) -> int:
    return load_library().awq_reserve(max_M, max_K, max_N, flags, stream)


def awq_shutdown() -> None:
    load_library().awq_shutdown()


def awq_linear_forward_decode_noalloc(x, qweight, qzeros, scales, bias, y, M, K, N, group_size,
                                      stream) -> int:
    """The decode forward with library-resident scratch: never allocates
    device memory (see include/awq_gb300.h for who needs this and its limits)."""
    return load_library().awq_linear_forward_decode_noalloc(x, qweight, qzeros, scales, bias, y,
                                                            M, K, N, group_size, stream)

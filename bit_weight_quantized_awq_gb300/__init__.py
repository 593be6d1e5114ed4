"""GB300 (sm_103a) AWQ W4A16 linear forward.

``y = x . dequant(W) + bias`` with W held as 4-bit codes packed eight per
int32 (nibble i of int32 j holds column 8j + i), per-group packed zero points
and fp16 scales -- the WQLinear layer of the Predibase Lorax "AWQ WQLinear"
page. The computation runs in hand-written CUDA kernels behind the C ABI in
``include/awq_gb300.h``; this package is the binding (``_binding``), a torch
wrapper (``layer``) and a seeded input generator (``synthetic``).
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    LIB_PATH,
    RESERVE_GIDX,
    RESERVE_SORTED,
    AWQError,
    Path,
    Status,
    awq_decode_tile_columns,
    awq_dequant,
    awq_dequant_gidx,
    awq_gemm_f16,
    awq_last_device_status,
    awq_linear_forward,
    awq_linear_forward_decode_noalloc,
    awq_finish_rows,
    awq_gidx_sort,
    awq_linear_forward_gidx,
    awq_linear_forward_sorted,
    awq_linear_forward_rows,
    awq_linear_forward_path,
    awq_pack,
    awq_path_supported,
    awq_permute_rows,
    awq_quantize_rtn,
    awq_reserve,
    awq_select_path,
    awq_forward_launches,
    awq_shutdown,
    awq_status_string,
    load_library,
)
from .layer import (AWQLinear, dequant, dequant_gidx, gidx_sort, linear_forward,  # noqa: F401
                    linear_forward_gidx, linear_forward_sorted, pack, prepare_act_order, quantize_rtn)

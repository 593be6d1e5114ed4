"""CPU oracle for the AWQ W4A16 linear forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library under
``bit_weight_quantized_awq_gb300`` never does, and shares no code with it.

Pinned functions (each one is checked by ``tests/test_oracle_pins.py``
against something other than itself):

* ``f64_to_f16_bits`` / ``f16_bits_to_f64`` -- IEEE binary16 written from its
  definition; pinned against numpy's correctly rounded conversion on every
  bit pattern and on every halfway case.
* ``unpack`` -- nibble i of int32 j holds column 8j + i; pinned by hand-packed
  hex fixtures in ``tests/golden/`` and by a one-hot placement test.
* ``dequant`` -- fp16_rn((q - z) * scale) per group of ``group_size`` input
  rows; pinned by exhaustive (q, z) x scale sweeps against exact rational
  arithmetic and by hand cases.
* ``forward`` -- fp64 sum over k of x * W16, plus bias; pinned by integer brute
  force on hand cases, the q == z identity, g = -1 vs g = K, scale doubling,
  per-group additivity and a library (numpy fp64 matmul) cross-check.
* ``dequant_gidx`` / ``forward_gidx`` -- the same with the group of input
  row k read from a table g_idx[k] ("act-order" grouping); pinned by equality
  with ``dequant`` / ``forward`` when g_idx[k] = k // g, by equivariance under
  a permutation of the rows, and by a constant table (one group) against
  ``dequant`` with g = K on that group's scales and zeros.
* ``pack`` -- the inverse of ``unpack``; pinned by the same hand-packed hex
  fixtures, a one-hot closed form for every nibble slot, and the two round
  trips with ``unpack``.
* ``quantize_rtn`` -- clamp(round_half_even(W / s) + z, 0, 15), packed;
  pinned by exact grid points (power-of-two scales), hand-computed ties and
  clamping cases, and quantize(dequant(q)) == q for arbitrary scales.
"""
from .oracle import (  # noqa: F401
    build,
    f64_to_f16_bits,
    f16_bits_to_f64,
    resolve_group,
    unpack,
    pack,
    quantize_rtn,
    dequant,
    forward,
    dequant_gidx,
    forward_gidx,
)

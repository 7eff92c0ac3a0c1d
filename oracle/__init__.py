"""fp64 CPU oracle for the hybrid sliding/global attention path.

TEST INFRASTRUCTURE: imported only by tests/, __graft_entry__.smoke() and the CPU legs of
bench.py. The product path never imports it. See oracle/core.py for the definitions,
their sources and the readings taken where the sources are silent.
"""
from .core import (GLOBAL, MAX_POSITIONS, SLIDING, Layer, Norms, attention, credited_prefill_flops,  # noqa: F401
                        decode_row, keys_values, layer_rows, normed_kv, normed_q, prefill, rms_norm, rope,
                        rope_inv_freq, rope_rotated_pairs, same_image, visible, with_window)

"""Oracle for the batched verify-window MoE decode step -- TEST INFRASTRUCTURE.

A plain, slow, fp64 CPU statement of what one verify window computes, used
only to check the CUDA path.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import or run anything in this
package; the library itself never does, and it shares no code, header, table
or helper with the CUDA sources.

Functions and the passage (or reading) each follows are listed in
``oracle/moe_window.py``.  Pins that tie each function to something other than
itself live in ``tests/test_oracle_*.py``.
"""
from .moe_window import (  # noqa: F401
    OQMat, OMoELayer, ODenseLayer,
    fp16_bits, unpack_codes, dequant, router, silu, expert_ffn, shared_ffn,
    group_rows, moe_row, moe_window, topk_margin,
    rmsnorm, dense_attention_len1, decoder_layer_row, stack_row,
)

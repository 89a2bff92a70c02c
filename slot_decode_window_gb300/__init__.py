"""GB300-native batched verify-window MoE decode step (C-ABI library + thin binding).

Import :mod:`slot_decode_window_gb300.binding` for the library calls; this
package's ``__init__`` deliberately loads nothing.
"""

"""Seeded synthetic THD packs for the CSA forward path.

This module only draws random numbers and shapes. It holds none of the
method's arithmetic (no compressed-length rule, no window or visibility
rule, no scoring, no attention), so that the CUDA path and the CPU oracle
can both consume the same inputs without sharing any computation.
"""

from .packs import (  # noqa: F401
    CONFIGS,
    LayerSpec,
    PackSpec,
    draw_layer_tensors,
    lognormal_lengths,
    make_cu_seqlens,
    pack_spec,
)

"""Seeded synthetic inputs for the paged-attention hot path.

This package draws input tensors and block layouts only.  It performs none of
the attention, RoPE or method-side rounding arithmetic: both the float64
oracle (``oracle/``) and the CUDA library consume what it produces.
"""

from .configs import (  # noqa: F401
    CONFIG_NAMES,
    DTYPE_CODES,
    TABLE_POISON,
    Workload,
    bf16_bits_from_f32,
    build_workload,
    describe,
    f16_bits_from_f32,
    make_config,
)

"""CPU float64 oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.

``oracle.fp8`` adds the FP8 (e4m3) quantisation and FP8 attention.
"""

from .attention import (  # noqa: F401
    attention,
    attention_backward,
    attention_band,
    attention_head,
    attention_rows,
    attention_varlen,
    combine_rows,
    decode,
    lse_merge,
    partial,
    split_partials,
    tree_combine,
    visible,
)
from . import fp8  # noqa: F401,E402

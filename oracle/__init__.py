"""FP64 CPU oracle for exact softmax attention -- test infrastructure only.

Importable from the test suite, the smoke check and the bench's CPU
baseline; never from the product path (`precision_numerics_gb300`).
"""
from . import int8  # noqa: F401
from .attention import (backward, backward_bhnd, delta, forward, forward_bhnd,  # noqa: F401
                        naive_bf16_backward, naive_bf16_forward, probabilities,
                        round_bf16, row_max, scores)

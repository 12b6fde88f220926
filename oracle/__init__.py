"""fp64 CPU oracles: fused linear cross-entropy and the generic chunked linear loss. TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and reference
legs may import this package. The CUDA library and its Python binding never
import it and share no code with it.

Parity status: every function is pinned. There is no "parity unpinned" entry.
tests/test_oracle_pins.py and tests/test_chunked_oracle_pins.py hold the
pins: torch fp64 autograd, finite differences, closed forms, invariants and
hand-derived golden values.
"""
from .flce_oracle import (  # noqa: F401
    REDUCTIONS, backward, check_targets, dlogits, forward, forward_rows,
    grad_hidden_rows, grad_weight_rows, row_gamma, row_terms, transformed_logits,
)
from .chunked_oracle import (  # noqa: F401
    chunked_linear_loss, cross_entropy_sum, weighted_mse,
)

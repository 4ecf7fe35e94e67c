"""fp64 CPU oracle (test infrastructure only; never on the product path).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. Every function is pinned by the CPU tests
in ``tests/test_oracle.py`` to closed forms, invariants, finite differences or
an independent library routine; no function is "parity unpinned".
"""

from .grpo_oracle import (  # noqa: F401
    IDENTITY,
    Transform,
    broadcast_advantage,
    grad_hidden,
    grad_weight,
    grpo_loss,
    logits_rows,
    logsumexp_rows,
    loss_fwd_bwd,
    rows_fwd_bwd,
    selective_logp,
    token_terms,
    token_weights,
)

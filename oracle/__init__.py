"""CPU oracle for the Sparse Delta Memory write/read op (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of
``bench.py`` may import this package.  The product path (``gated_delta_rule_factor_gb300``)
never does; the two share no code.
"""
from .sdm_oracle import *  # noqa: F401,F403
from .sdm_oracle import __all__  # noqa: F401

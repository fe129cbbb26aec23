"""CPU fp64 oracle for MSA (MiniMax-style sparse attention) training.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may use it.  It shares no code with the CUDA path.
"""
from .msa_oracle import (  # noqa: F401
    OracleParams,
    pooled_proxy_scores,
    select_blocks,
    select_from_pooled,
    msa_reference,
    row_reference,
    effective_flops,
)

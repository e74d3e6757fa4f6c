"""CPU oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does.
"""
from .oracle import (  # noqa: F401
    E4M3_TABLE, bf16_to_f64, e4m3_to_f64, decode, token_request, token_position,
    valid_slots, attend, partial, combine_partials, sparse_mla_decode, run_workload,
)

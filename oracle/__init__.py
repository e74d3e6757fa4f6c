"""CPU oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does.
"""
from .oracle import (  # noqa: F401
    E4M3_TABLE, E2M1_TABLE, PACKED_ROW_BYTES, bf16_to_f64, e4m3_to_f64, ue8m0_to_f64, decode,
    decode_rows, decode_packed_fp8_rows, decode_nvfp4_rows, token_request, token_position,
    valid_slots, attend, partial, combine_partials, sparse_mla_decode, run_workload,
)

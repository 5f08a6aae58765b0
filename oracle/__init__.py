"""Double-precision CPU oracle for paged gated-MLA decode.

TEST INFRASTRUCTURE ONLY: tests/, the smoke check in __graft_entry__ and the
CPU-baseline leg of bench.py may import this package; the product library never
does.  It shares no code with the CUDA path.
"""
from .oracle import (  # noqa: F401
    attend_rows,
    gate_sigmoid,
    kv_append,
    lse_merge,
    mla_decode_reference,
    plan_splits,
    split_budget,
)

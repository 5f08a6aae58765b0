"""Double-precision CPU oracle for paged gated-MLA decode.

TEST INFRASTRUCTURE ONLY: tests/, the smoke check in __graft_entry__ and the
CPU-baseline leg of bench.py may import this package; the product library never
does.  It shares no code with the CUDA path.
"""
from .oracle import (  # noqa: F401
    E4M3_MAX,
    attend_rows,
    dequantize_query_rows,
    e4m3_decode,
    e4m3_encode,
    gate_sigmoid,
    kv_append,
    kv_append_e4m3,
    lse_merge,
    mla_decode_e4m3_reference,
    mla_decode_reference,
    plan_splits,
    plan_splits_uniform,
    quantize_query_rows,
    query_scale_exponent,
)

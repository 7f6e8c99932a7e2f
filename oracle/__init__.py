"""Plain CPU oracle of the weight-streaming decode path (float64).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg. The product library does not import, link or
call anything here, and nothing here uses the product library.

Every function is pinned by CPU tests against closed forms, invariants,
special cases and brute force (tests/test_oracle_*.py).
"""
from .primitives import (  # noqa: F401
    argmax_lowest,
    bf16_bits_of,
    causal_prefill_attention,
    gemv,
    gemv_q4,
    gqa_decode_attention,
    project_rows,
    q4_dequant,
    q4_unpack,
    rmsnorm,
    rope,
    round_to_bf16,
    silu,
    softmax,
    swiglu,
    widen,
)
from .decoder import OracleDecoder, generate  # noqa: F401

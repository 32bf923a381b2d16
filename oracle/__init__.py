"""CPU oracle for the routing + dispatch + grouped-GEMM path.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The product library never imports it.
"""
from .oracle import (  # noqa: F401
    build_oracle,
    topk,
    renorm_gates,
    select_biased,
    gates_at,
    histogram,
    permutation,
    rank_base,
    gather,
    grouped_gemm,
    grouped_gemm_parallel,
    gemm_entry,
    expert_of_row,
    route,
    combine,
    router_logits,
    swiglu,
    round_bf16,
)

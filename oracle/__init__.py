"""CPU oracle for the fine-grained MoE layer forward -- TEST INFRASTRUCTURE.

A plain, slow, fp64 restatement of what the pages define, used only to check
the CUDA path.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the product package never does,
and this package never imports the product package.  It shares no code with
the CUDA path: its only common dependency is the seeded input generator in
``synth``, which holds no arithmetic of the method.

Every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against brute force, closed forms and the
invariants the pages fix.  Parts with no such pin would say "parity unpinned"
here; the K3 latent composition is pinned only through its reduction to the K2
form (identity projections), which is stated in that test.
"""
from .moe_oracle import (  # noqa: F401
    ROUTED_SCALING_FACTOR,
    bf16_bits_to_f64,
    e4m3_to_f64,
    FP8_BLOCK,
    dequant_fp8_blocks,
    sigmoid,
    silu,
    round_f32,
    biased_scores_f32,
    group_scores_f32,
    select_experts,
    selection_gaps,
    router_weights,
    router_from_logits,
    router_from_x,
    dense_gates,
    aux_free_bias_update,
    quantile_bias_update,
    permute,
    combine,
    swiglu_expert,
    moe_layer,
    moe_layer_tokens,
    moe_layer_tokens_fp8,
)

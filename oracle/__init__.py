"""CPU oracle of the W4A16 fused MoE feed-forward -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use it.
"""
from .moe_oracle import (  # noqa: F401
    GROUP_SIZE,
    bf16_to_f64,
    dequantize,
    dequantize_ct,
    dequantize_g_idx,
    expert_dense,
    expert_ffn,
    expert_hidden,
    moe_align,
    moe_forward,
    roofline_bytes_per_expert,
    route,
    silu,
    unpack_codes,
    unpack_codes_ct,
)

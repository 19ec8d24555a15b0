"""CPU oracle of the block-FP8 mixture-of-experts layer forward.

TEST INFRASTRUCTURE ONLY: a plain, slow, obviously correct numpy statement of
what the layer computes, used to check the CUDA path. Only the tests, the smoke
check and the CPU-baseline leg of the benchmark may import it; the library
never does, and it imports nothing from the library.

Pins (tests/test_oracle_pins.py) tie every function here to something other
than itself: format definitions, closed forms, brute force on tiny inputs,
exact rational arithmetic, library conversions, and layer invariants.
"""

from .formats import (  # noqa: F401
    E4M3_MAX,
    E4M3_VALUES,
    bf16_bits,
    bf16_from_bits,
    bf16_round,
    e4m3_decode,
    e4m3_encode,
    fma_f32,
    pow2_ceil,
    ue8m0_to_f32,
)
from .moe_ref import (  # noqa: F401
    ALIGN,
    CLAMP_AFTER_SILU,
    CLAMP_BEFORE_SILU,
    CLAMP_NONE,
    GROUP,
    NUMERICS_DIVIDE,
    NUMERICS_RECIPROCAL,
    SCALE_FLOOR,
    SCALE_FP32,
    SCALE_FP32_POW2,
    SCALE_UE8M0,
    align,
    batched_forward,
    block_gemm,
    expert_rows,
    group_scale,
    moe_forward,
    quant_1x128,
    scale_bytes,
    swiglu,
    topk_reduce,
    weight_scales_f32,
)

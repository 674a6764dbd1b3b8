"""CPU oracle for the small-batch MoE decode layer step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA library never calls into it and shares no code with it; the product path
fails loudly when its CUDA extension is missing instead of falling back here.

Everything is float64 numpy. Inputs arrive as the exact bit patterns the GPU
consumes (bf16 as uint16, NVFP4 codes and e4m3 scales as uint8) and are widened
exactly, so the oracle sees the same numbers as the kernels.

Modules:
  moe_oracle -- router GEMV, top-k + renormalised weights, SwiGLU experts,
                weighted combine + shared expert + residual, RMSNorm.
  nvfp4      -- e2m1 / e4m3 decoding and NVFP4 block dequantisation.
"""

from .moe_oracle import (  # noqa: F401
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    router_logits,
    topk_renorm,
    route,
    silu,
    expert_swiglu,
    moe_layer,
    rmsnorm,
    stack_layer_input,
    topk_margin,
    expert_union,
)
from .nvfp4 import e2m1_value, e4m3_value, dequant_nvfp4_rows  # noqa: F401

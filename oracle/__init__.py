"""CPU oracle for the small-batch MoE decode layer step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA library never calls into it and shares no code with it; the product path
fails loudly when its CUDA extension is missing instead of falling back here.

Two independent restatements of the same definitions, both float64:
  cpp        -- the oracle proper: plain C++ loops (``moe_oracle_ref.cpp``, built
                by ``build.py`` into a shared library, OpenMP over independent
                output elements), loaded through ctypes. The GPU parity tests and
                the bench's CPU baseline use it.
  moe_oracle -- a numpy restatement (router GEMV, selection, SwiGLU experts,
                combine, RMSNorm), plus ``nvfp4`` for e2m1 / e4m3 decoding and
                the NVFP4 and FP8 block dequantisation. The
                tests run every pin against both and cross-check the two on random
                layers.

Inputs arrive as the exact bit patterns the GPU consumes (bf16 as uint16, NVFP4
codes and e4m3 scales as uint8) and are widened exactly, so the oracle sees the
same numbers as the kernels.
"""

from .moe_oracle import (  # noqa: F401
    SCORE_SIGMOID_BIAS,
    SCORE_SOFTMAX,
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    router_logits,
    topk_renorm,
    select,
    sigmoid_bias_select,
    route,
    silu,
    expert_swiglu,
    moe_layer,
    rmsnorm,
    stack_layer_input,
    topk_margin,
    expert_union,
)
from .nvfp4 import e2m1_value, e4m3_value, dequant_nvfp4_rows, dequant_fp8_block  # noqa: F401

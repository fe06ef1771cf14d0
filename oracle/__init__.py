"""CPU oracle for the NF4-QLoRA linear layer.  Test infrastructure only: the
product path never imports it (see ``qlora_oracle`` for what it computes)."""
from .qlora_oracle import (  # noqa: F401
    BLOCK, NF4_CODE, ZERO_CODE, bf16_bits, bf16_round, code_midpoints,
    dequantize_nf4, lora_backward, lora_forward, lora_scale, merged_weight, merged_weight_bf16,
    nearest_code, quantize_nf4, swiglu_backward, swiglu_forward, swiglu_mlp_backward,
    swiglu_mlp_forward, unpack_codes,
)

"""NF4-QLoRA fused linear layer for B300 (sm_103a): C-ABI library + thin binding."""

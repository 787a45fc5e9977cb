"""GB300-native APEX-1 attention block (RoPE + GQA + causal/sliding-window SDPA)."""

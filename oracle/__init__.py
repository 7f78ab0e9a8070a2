"""CPU oracle for the MXFP4 MoE layer (test infrastructure only; see mxfp4_moe_oracle)."""

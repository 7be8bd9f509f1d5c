"""CPU oracle for the MoE layer forward: test infrastructure only (see moe_oracle)."""

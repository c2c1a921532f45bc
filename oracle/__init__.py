"""CPU oracle of the NVFP4 MoE forward (test infrastructure only; see nvfp4_oracle)."""

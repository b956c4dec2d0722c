"""CPU oracle for the NVFP4 W4A4 linear layer (test infrastructure only)."""

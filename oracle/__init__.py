"""CPU oracle for the MoE FFN layer: test infrastructure, never called by the CUDA library."""

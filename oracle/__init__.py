"""CPU oracle for the MoE dispatch + expert-GEMM path (test infrastructure only)."""

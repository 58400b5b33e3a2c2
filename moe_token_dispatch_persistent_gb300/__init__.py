"""GB300-native MoE token dispatch + expert GEMM in one persistent kernel."""

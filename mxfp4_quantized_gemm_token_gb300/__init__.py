"""GB300-native quantized scaled GEMM and routed fused MoE (placeholder; the
binding is filled in with the CUDA library)."""

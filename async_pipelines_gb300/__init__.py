"""GB300-native persistent warp-specialized bf16 GEMM with tile stream-out."""

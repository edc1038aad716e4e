"""GB300-native single-precision GEMM (placeholder; the binding lands with the C-ABI)."""

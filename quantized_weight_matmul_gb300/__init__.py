"""GB300-native quantized-weight matmul (placeholder until the binding lands)."""

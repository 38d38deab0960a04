"""GB300-native low-bit quantized matrix-vector product (binding placeholder)."""

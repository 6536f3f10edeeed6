"""GB300-native verify matmul for speculative decoding (placeholder; binding follows)."""

"""GB300-native low-bit KV-cache quantization with fused split-KV decode attention."""

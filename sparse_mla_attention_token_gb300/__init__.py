"""GB300-native sparse MLA prefill forward (DeepSeek-V4, K == V, D = 512)."""

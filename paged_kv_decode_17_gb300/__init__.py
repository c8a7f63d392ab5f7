"""GB300-native exact softmax attention over a paged bf16 KV cache."""

"""GB300-native decode attention over a static KV cache."""

"""GB300-native speculative-decoding verification (vectorised rejection sampler)."""

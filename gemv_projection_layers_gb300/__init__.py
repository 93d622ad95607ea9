"""GB300-native dense projections (out = x @ W.T) behind a C ABI."""

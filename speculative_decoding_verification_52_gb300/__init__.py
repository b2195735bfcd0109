"""GB300-native batched draft-token verification for speculative decoding."""

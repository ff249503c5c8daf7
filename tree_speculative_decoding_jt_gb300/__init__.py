"""GB300-native hot path of JetSpec-style tree speculative decoding."""

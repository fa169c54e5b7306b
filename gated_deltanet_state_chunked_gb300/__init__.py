"""GB300-native Gated DeltaNet tail-replay state rebuild."""

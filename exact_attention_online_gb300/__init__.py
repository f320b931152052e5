"""GB300-native exact attention (online softmax forward, recompute backward)."""

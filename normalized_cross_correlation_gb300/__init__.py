"""GB300-native normalized cross-correlation (NCC) template matching."""

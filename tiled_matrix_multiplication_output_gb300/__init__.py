"""GB300-native output-stationary tiled matrix multiply (placeholder)."""

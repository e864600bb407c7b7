"""GB300-native dense matrix multiplication (placeholder; binding follows)."""

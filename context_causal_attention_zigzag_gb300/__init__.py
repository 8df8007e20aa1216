"""GB300-native context-parallel zigzag causal attention (placeholder, filled below)."""

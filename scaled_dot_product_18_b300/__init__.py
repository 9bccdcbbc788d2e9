"""B300-native multi-head scaled dot-product attention forward (placeholder binding)."""

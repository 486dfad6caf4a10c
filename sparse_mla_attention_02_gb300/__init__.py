"""GB300-native sparse MLA attention forward (placeholder; binding follows)."""

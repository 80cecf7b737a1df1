"""GB300-native paged KV-cache hot path (placeholder; binding follows)."""

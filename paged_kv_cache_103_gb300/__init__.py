"""GB300-native paged KV-cache decode attention (sm_103a)."""

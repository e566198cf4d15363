"""GB300-native W4A16 routed mixture-of-experts layer (placeholder, filled in below)."""

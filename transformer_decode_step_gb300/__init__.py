"""GB300-native transformer decode step (binding filled in with the library)."""

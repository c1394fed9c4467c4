"""GB300-native image resize (placeholder; the binding is added with the library)."""

"""GB300-native paged decode attention (placeholder; binding added with the library)."""

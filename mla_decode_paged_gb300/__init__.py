"""GB300-native MLA paged decode (placeholder; binding added with the library)."""

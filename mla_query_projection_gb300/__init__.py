"""GB300-native decode-step MLA query path (placeholder; binding added with the library)."""

"""GB300-native CSA2 sparse decode attention (placeholder; binding added with the library)."""

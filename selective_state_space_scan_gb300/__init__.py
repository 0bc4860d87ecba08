"""GB300-native selective scan (placeholder; binding added with the CUDA library)."""

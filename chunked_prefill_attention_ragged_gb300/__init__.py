"""GB300-native MLA ragged prefill (placeholder; binding added with the C-ABI)."""

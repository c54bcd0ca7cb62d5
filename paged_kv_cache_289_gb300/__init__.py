"""libpagedkv Python binding (filled in with the C-ABI library)."""

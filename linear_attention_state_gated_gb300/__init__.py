"""GB300-native segment scan and state composition for position-independent
caching of hybrid linear-attention models (HYPIC)."""

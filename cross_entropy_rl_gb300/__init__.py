"""GB300-native fused linear log-probability (see ``binding`` for the calls)."""

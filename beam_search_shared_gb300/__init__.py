"""GB300-native shared-prefix (cascade) beam decode attention."""

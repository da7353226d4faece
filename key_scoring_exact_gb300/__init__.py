"""GB300-native index chain: paged FP8 key scoring and exact top-k selection."""

"""GB300-native channels-last GroupNorm(+SiLU)."""

"""GB300-native block-sparse masked attention forward (Splash-style)."""

"""GB300-native device-wide prefix sum (single-pass decoupled look-back)."""

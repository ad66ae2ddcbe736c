"""GB300-native draft-head argmax library (Python binding; filled in below)."""

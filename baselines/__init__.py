"""Comparison baselines timed beside the library: the pages' own dense-operation
formulations, in plain PyTorch. Not part of the library."""

"""GB300-native batched constrained logits sampler.

The compute path is the CUDA library ``libclsample.so`` (built from ``csrc/``); the
Python side only marshals arguments.  Importing the package does not load the
library: ``sampler.Sampler`` does, and it raises if the library is missing.
"""

__all__ = ["workloads", "sampler"]

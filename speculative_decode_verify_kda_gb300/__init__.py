"""GB300-native speculative-verify walk through a Kimi-Delta-Attention layer.

The compute path is the CUDA library built from ``csrc/`` (C ABI declared in
``include/kda_spec.h``); ``binding`` marshals torch tensors into it.  Importing
this package loads nothing; ``binding`` raises if the library is missing.
"""
__version__ = "0.1.0"

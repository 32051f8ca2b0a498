"""Deterministic gated BF16 FFN for GB300 (sm_103a): Python binding of libdetffn.

The compute path is the C-ABI library ``libdetffn.so`` built from ``csrc/``;
this package only marshals arguments (tensor pointers, sizes, the current CUDA
stream).  Importing the package does not load the library; the first call
does, and raises if the library is missing -- there is no CPU fallback.
"""

"""GB300 (sm_103a) library for the Gated Delta Rule linear-attention layer over a slot pool.

The compute path is the C-ABI shared library ``libgdn.so`` built from ``csrc/``;
``binding`` wraps it with ctypes (argument marshalling only).  ``synth`` draws
the seeded synthetic inputs.  Importing the package does not load the CUDA
library; the first call into ``binding`` does, and fails loudly if it is missing.
"""

"""GB300-native tree verification for lossless speculative decoding.

The compute lives in ``libspectree.so`` (hand-written sm_103a CUDA kernels
behind a C ABI, declared in ``include/spec_tree.h``).  ``binding`` marshals
torch tensors into those calls; ``synth`` draws seeded synthetic inputs.
Importing this package does not load the CUDA library; the first call through
``binding`` does, and fails loudly if it is missing.
"""
__version__ = "0.1.0"

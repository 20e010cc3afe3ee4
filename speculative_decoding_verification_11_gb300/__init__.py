"""GB300-native verification step of speculative decoding.

The compute path is libspecverify.so (hand-written sm_103a CUDA, C ABI in
include/specverify.h).  ``binding`` exposes its entry points under the same
names; ``api`` adds output/workspace allocation through torch; ``workloads``
builds the seeded synthetic inputs.  Importing the package does not load the
library; the first call does, and fails loudly if it was not built.
"""
__all__ = ["api", "binding", "build", "workloads"]

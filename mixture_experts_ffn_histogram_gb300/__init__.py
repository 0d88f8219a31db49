"""GB300-native (sm_103a) sparse mixture-of-experts expert block.

The compute lives in libmoe.so (hand-written CUDA: routing histogram,
permute, tcgen05 grouped GEMMs with fused SwiGLU, combine, and every
backward), declared in ``include/moe.h``.  ``binding`` wraps each C entry
point under the same name; ``block.MoEBlock`` strings the calls together over
caller-owned device buffers; ``inputs`` draws the seeded synthetic workloads.
Importing this package does not load the library; the first call does, and
fails loudly if it has not been built.
"""
__all__ = ["binding", "block", "inputs"]

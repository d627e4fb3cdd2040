"""GB300-native hot path of one DSpark speculative-decoding cycle.

Markov/RNN-head drafting, lossless rejection-sampling verification and the
confidence scheduler, as hand-written sm_103a CUDA kernels behind the C ABI of
``include/dspark.h`` (``libdspark.so``).  ``binding`` is the thin Python
marshalling layer; ``synth`` draws the seeded synthetic inputs.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "binding"]

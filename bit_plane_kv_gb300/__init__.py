"""GB300 (sm_103a) implementation of the Fathom variable-depth bit-plane key
scan for top-k sparse decode attention.

The computation lives in libfathom (CUDA, C ABI in include/fathom.h);
``binding`` is its thin Python face, ``synth`` draws seeded synthetic inputs,
``build`` compiles the library in-tree.
"""
from . import binding  # noqa: F401

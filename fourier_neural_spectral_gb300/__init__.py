"""libfnospec: the FNO 2D spectral-convolution layer on one GB300 GPU.

The CUDA library (``libfnospec.so``, built in-tree by ``build.py``) is the
product; ``fourier_neural_spectral_gb300.fnospec`` is its thin ctypes binding
(import it explicitly).  ``synth`` generates the seeded synthetic inputs.
Importing this package does not load the CUDA library; the first call into
``fnospec`` does, and raises if it is missing.
"""
from . import synth  # noqa: F401

__all__ = ["synth"]

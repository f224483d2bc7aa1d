"""GB300-native (sm_103a) Gated DeltaNet sublayer: CUDA kernels behind a C ABI (``libgdn.so``).

The Python surface is a thin ctypes binding over the C entry points declared in
``include/gdn.h`` (same names); it only marshals arguments.  Importing this package does not load
the library; the first call does, and fails loudly when the CUDA library is missing.
"""
from .synth import Geometry, QWEN_GDN  # noqa: F401

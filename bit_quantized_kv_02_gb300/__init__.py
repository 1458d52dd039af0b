"""GB300-native group-wise integer KV-cache quantization and quantized decode attention.

The compute path lives in libkvq.so (CUDA kernels for sm_103a behind the C ABI
of include/kvq.h); ``kvq`` is its thin ctypes binding and ``synth`` holds the
seeded synthetic input generators.  ``build.build()`` compiles the library.
"""
from . import build  # noqa: F401

"""libkq: GB300-native decode-time products against GGUF k-quant weights.

The compute lives in libkq.so (CUDA for sm_103a, C ABI in include/kq.h);
``kq`` is its thin ctypes binding and ``synth`` the seeded synthetic inputs.
"""
from . import kq  # noqa: F401

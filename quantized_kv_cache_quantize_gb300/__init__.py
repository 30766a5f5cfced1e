"""GB300-native Jensen-bias-corrected low-bit KV-cache chunk attention.

The compute path is libkvq.so (CUDA, sm_103a); ``kvq`` is its ctypes binding.
"""
from . import kvq  # noqa: F401
from .kvq import (CORR_NONE, CORR_TAYLOR, KVCache, KVQError, attention_corrected,  # noqa: F401
                  attention_mass, quantize_append, rotate)

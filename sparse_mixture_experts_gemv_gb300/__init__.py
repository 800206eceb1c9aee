"""GB300-native sparse mixture-of-experts layer (router + top-k + shared expert).

The layer runs in libmoe.so (hand-written sm_103a CUDA, C ABI in
include/moe_layer.h); this package is its ctypes binding plus a small owner
object. The library is loaded on first use; if it has not been built, that
first call raises ImportError (there is no fallback implementation).
"""
from ._native import *  # noqa: F401,F403  (C names: moe_layer_create, moe_layer_forward, ...)
from ._native import load  # noqa: F401
from .layer import MoeLayer, weights_from_raw  # noqa: F401
from .lmhead import LmHead  # noqa: F401

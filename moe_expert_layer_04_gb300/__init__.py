"""GB300-native routed Mixture-of-Experts layer (DeepSeek-V4 style) on one GPU.

The compute lives in libmoe.so (CUDA kernels for sm_103a behind the C ABI of
include/moe.h); `_lib` binds it, `layer` sequences its calls, `workloads`
draws seeded synthetic inputs.
"""
from . import _lib  # noqa: F401
from ._lib import build, load  # noqa: F401

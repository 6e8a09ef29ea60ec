"""GB300-native blockwise causal attention with log-sum-exp merging for ring /
zigzag context parallelism over C virtual ranks on one GPU.

The compute path is libcpattn.so (CUDA, sm_103a) behind the C ABI in
include/cpattn.h; ``ops`` is its thin Python binding.
"""
from .ops import *  # noqa: F401,F403
from .ops import __all__  # noqa: F401

"""GB300-native training-mode normalization forward/backward.

The compute lives in ``libgbnorm.so`` (hand-written CUDA for sm_103a, C ABI
in ``include/gbnorm.h``); ``bwd_bn_pass_gb300.gbnorm`` is its ctypes binding.
Importing this package loads nothing: the library is opened on first use.
"""

__version__ = "0.1.0"

"""Float64 CPU oracle for training-mode normalization forward/backward.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plainly written
reference that the CUDA library is checked against.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it.  The library (``bwd_bn_pass_gb300``) never
imports it, and the two share no code: no kernels, helpers, constants or
pre/post-processing.  Inputs are the exact stored values widened to float64;
nothing is rounded to a storage type inside the oracle.

Every function is written from the pages it cites and pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_pins.py`` against things other
than itself: PyTorch float64 autograd (an independent implementation),
central finite differences, closed-form invariants and exact rational
arithmetic.  No function here is "parity unpinned".
"""

from .bn import (
    batch_norm_forward_train,
    batch_norm_apply,
    batch_norm_backward,
    batch_norm_act_forward_train,
    batch_norm_act_backward,
    batch_norm_nhwc_forward_train,
    batch_norm_nhwc_backward,
    activation,
    activation_gate,
    ACT_NONE,
    ACT_RELU,
    ACT_LEAKY_RELU,
)
from .rmsnorm import rms_norm_rstd, rms_norm_forward, rms_norm_backward
from .layernorm import (
    dropout_add,
    layer_norm_saved_stats,
    layer_norm_forward,
    fused_bias_dropout_add_layer_norm_forward,
    layer_norm_backward,
    fused_bias_dropout_add_layer_norm_backward,
    layer_norm_backward_saved_z,
)

__all__ = [
    "batch_norm_forward_train",
    "batch_norm_apply",
    "batch_norm_backward",
    "batch_norm_act_forward_train",
    "batch_norm_act_backward",
    "batch_norm_nhwc_forward_train",
    "batch_norm_nhwc_backward",
    "activation",
    "activation_gate",
    "rms_norm_rstd",
    "rms_norm_forward",
    "rms_norm_backward",
    "dropout_add",
    "layer_norm_saved_stats",
    "layer_norm_forward",
    "fused_bias_dropout_add_layer_norm_forward",
    "layer_norm_backward",
    "fused_bias_dropout_add_layer_norm_backward",
    "layer_norm_backward_saved_z",
]

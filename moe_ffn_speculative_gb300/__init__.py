"""GB300-native (sm_103a) MoE-FFN layer forward for DFlash/DSpark draft models.

The compute lives in ``libmoe_gb300.so`` (hand-written CUDA, C ABI declared in
``include/moe.h``); ``moe_ffn_speculative_gb300.ops`` marshals torch tensors
into those calls.
"""
from .synthetic import CONFIGS, LayerConfig, make_inputs  # noqa: F401

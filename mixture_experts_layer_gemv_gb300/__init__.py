"""GB300-native (sm_103a) forward pass of a DeepSeek-style MoE layer.

The compute lives in libmoe_gb300.so (C ABI: include/moe.h); `binding` is its thin
Python front end and `synth` makes seeded synthetic layers and tokens.
"""
from .synth import MoEConfig, WORKLOADS  # noqa: F401

__all__ = ["MoEConfig", "WORKLOADS", "binding", "synth", "build"]

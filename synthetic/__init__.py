"""Seeded synthetic inputs for the MoE layer.

This package holds shapes and random draws only. It contains none of the
layer's arithmetic: both the CPU oracle and the CUDA path take their inputs
from here and from nowhere else.
"""
from .configs import CONFIGS, MoEConfig, get_config, small_variant
from .gen import make_inputs, normal_bf16, normal_f32, bf16_bits_to_f32

__all__ = ["CONFIGS", "MoEConfig", "get_config", "small_variant", "make_inputs",
           "normal_bf16", "normal_f32", "bf16_bits_to_f32"]

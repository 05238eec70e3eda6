"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This package only draws random numbers and shapes them into the cached
activations, weights and adapter states of a layer; it computes no gradient.
"""
from . import rng
from .configs import CONFIGS, DECODE, SEQ512, STACK2048, TINY, LayerConfig
from .inputs import attention_rows, layer_inputs, layer_inputs_sample, row_slice, stack_dout, vector

__all__ = ["rng", "CONFIGS", "DECODE", "SEQ512", "STACK2048", "TINY", "LayerConfig",
           "attention_rows", "layer_inputs", "layer_inputs_sample", "row_slice", "stack_dout", "vector"]

"""Seeded synthetic inputs for paged decode attention.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It draws random numbers, lays out block tables and context
lengths, and packs bf16 values; it holds none of the attention arithmetic and
none of the FP8 codec.
"""
from .gen import (  # noqa: F401
    DecodeCase,
    bf16_bits_from_f32,
    bf16_bits_to_f32,
    normal_bf16_bits,
    fp8_tile_scales,
    int8_tile_params,
    tiny_case,
    llama8b_layer_case,
    mixed_prefix_case,
    long_context_case,
    fp8_shared_case,
    random_case,
    CONFIG_BUILDERS,
)

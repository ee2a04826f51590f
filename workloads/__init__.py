"""Seeded synthetic inputs for the routed-expert MoE layer.

This package is the one thing the CUDA path, the oracle, the tests and the
bench share.  It draws random inputs and stores them in the formats the layer
consumes; it computes nothing the layer computes.
"""
from .generate import (  # noqa: F401
    CONFIGS,
    LayerConfig,
    Weights,
    Tokens,
    make_weights,
    make_tokens,
    make_hash_table,
    bf16_bits_from_f32,
    bf16_bits_to_f32,
    encode_mxfp4_rows,
    encode_nvfp4_rows,
    encode_fp8_tiles,
)

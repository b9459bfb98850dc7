"""Seeded synthetic inputs for MLA tree-verify attention.

This package only draws random inputs (queries, latent KV rows, draft
trees, slot placements). It holds none of the attention arithmetic and
none of the index/mask construction: both the CPU oracle and the CUDA
path consume what it produces.
"""

from .gen import (  # noqa: F401
    CONFIGS,
    D_QK,
    D_V,
    VerifyInputs,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    SPARSE_DECODE,
    AcceptInputs,
    IndexerInputs,
    RelocateInputs,
    make_accept_inputs,
    make_config,
    make_indexer_inputs,
    make_inputs,
    make_relocate_inputs,
    make_sparse_decode,
)

"""Ternary projection linears (weights in {-1, 0, +1}, one fp32 scale per
output row) for B300 (sm_103a).

The CUDA library and its Python binding live in ``bit_matvec_ternary_b300.tl``;
``bit_matvec_ternary_b300.synth`` draws seeded synthetic inputs.  Importing
the package itself loads nothing.
"""
__version__ = "0.1.0"

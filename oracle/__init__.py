"""CPU float64 oracle of the latent-MoE layer tail (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU timing leg of ``bench.py`` use
this package; the CUDA path never imports it.
"""
from .codecs import e2m1_decode, e4m3_decode, e4m3_encode, unpack_e2m1  # noqa: F401
from .model import (bf16_round, dequant_fp8_blocks, dequant_mx, dequant_nvfp4,  # noqa: F401
                   latent_inputs, permutation, quant_mx, quant_per128, rmsnorm, route, silu,
                   swiglu_mlp, tail)

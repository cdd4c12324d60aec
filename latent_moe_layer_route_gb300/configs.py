"""Workload definitions for the latent-MoE layer tail.

The five named workloads are the synthetic shapes the tail is checked and timed on:
a tiny oracle case, two decode batches and two prefill batches (one with NVFP4 routed
weights).  Widths follow the Kimi K3 latent-MoE layout described in the vLLM pull request
"Fuse BF16 shared experts into latent MegaMoE tail" (Summary): the routed experts work in
the 3584-wide latent space and the shared expert in the 7168-wide hidden space.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

FMT_FP8 = "fp8"      # e4m3 codes with one fp32 scale per 128x128 block
FMT_NVFP4 = "nvfp4"  # e2m1 codes, e4m3 scale per 16 K-elements, fp32 per-matrix scale
FMT_MXFP8 = "mxfp8"  # e4m3 codes, one power-of-two (UE8M0) scale per 32 K-elements
FMT_W4A4 = "nvfp4_w4a4"  # NVFP4 weights and NVFP4 activations (e2m1, e4m3 scale per 16)


@dataclass(frozen=True)
class TailConfig:
    name: str
    M: int                      # tokens
    E: int                      # routed experts
    topk: int
    I: int                      # routed expert intermediate width
    H: int = 7168               # hidden width (shared expert input, tail output)
    L: int = 3584               # latent width (routed expert input/output)
    Is: int = 2048              # shared expert intermediate width
    routed_fmt: str = FMT_FP8
    router: str = "normal"      # "normal" | "bias_normal" | "zipf"
    seed: int = 0
    eps: float = 1e-6

    def with_(self, **kw) -> "TailConfig":
        return replace(self, **kw)


TINY_M4 = TailConfig("tiny_m4_e16_k4", M=4, E=16, topk=4, I=512, seed=0)
DECODE_M16 = TailConfig("decode_m16_e64_k8_fp8", M=16, E=64, topk=8, I=1024, seed=1)
DECODE_M128 = TailConfig("decode_m128_e64_k8_fp8_biased", M=128, E=64, topk=8, I=1024,
                         router="bias_normal", seed=2)
PREFILL_M4096 = TailConfig("prefill_m4096_e64_k8_fp8_zipf", M=4096, E=64, topk=8, I=1024,
                           router="zipf", seed=3)
PREFILL_M8192_NVFP4 = TailConfig("prefill_m8192_e128_k8_nvfp4", M=8192, E=128, topk=8,
                                 I=1024, routed_fmt=FMT_NVFP4, seed=4)

ALL = [TINY_M4, DECODE_M16, DECODE_M128, PREFILL_M4096, PREFILL_M8192_NVFP4]

# The power-of-two-scale variants (MXFP8 routed weights and activations) of the decode and
# prefill workloads, for comparison with the FP8 128x128-block path on the same shapes.
DECODE_M16_MX = DECODE_M16.with_(name="decode_m16_e64_k8_mxfp8", routed_fmt=FMT_MXFP8)
PREFILL_M4096_MX = PREFILL_M4096.with_(name="prefill_m4096_e64_k8_mxfp8_zipf",
                                       routed_fmt=FMT_MXFP8)
# The FP4 x FP4 variant of the NVFP4 prefill workload: the same weights, activations
# quantised to NVFP4 too, so the routed GEMMs run block-scaled at the FP4 rate.
DECODE_M16_W4A4 = DECODE_M16.with_(name="decode_m16_e64_k8_nvfp4_w4a4", routed_fmt=FMT_W4A4)
PREFILL_M8192_W4A4 = PREFILL_M8192_NVFP4.with_(name="prefill_m8192_e128_k8_nvfp4_w4a4",
                                               routed_fmt=FMT_W4A4)
VARIANTS = [DECODE_M16_MX, PREFILL_M4096_MX, DECODE_M16_W4A4, PREFILL_M8192_W4A4]
BY_NAME = {c.name: c for c in ALL + VARIANTS}

# Small shapes (every width one or two 128-tiles) used by fast parity and oracle tests.
SMALL = TailConfig("small_h256_l256_e4_k2", M=6, E=4, topk=2, I=128, H=256, L=256, Is=128,
                   seed=11)

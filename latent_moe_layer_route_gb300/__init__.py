"""GB300-native latent-MoE layer tail (routed FP8/NVFP4 experts in the latent space,
RMSNorm + up-projection, BF16 shared expert) behind a C-ABI library."""
from . import configs  # noqa: F401

"""Seeded synthetic inputs and weights for the latent-MoE layer tail.

This module draws random numbers and stores them in the formats the tail consumes.  It
holds none of the tail's own arithmetic: the offline weight quantisers below only turn
the drawn float weights into the stored FP8 / NVFP4 formats (the tail receives weights
already quantised), and the float -> e4m3 code step uses PyTorch's own cast.

Draw recipe (numpy ``default_rng``; two independent streams so that token inputs and
weights can vary separately):

* activations stream ``default_rng([seed, 0])``: x[M,H], z[M,L] ~ N(0,1) rounded to bf16;
  router logits[M,E] ~ N(0,1) in fp32; then the per-expert router bias (see ``router``).
* weights stream ``default_rng([seed, 1])``: gamma[L] ~ U(0.5,1.5) (bf16); W13 expert by
  expert, W2 expert by expert, shared Ws13, shared Ws2, up-projection W_up, every weight
  ~ N(0, 1/fan_in) in fp32 before its storage format is applied.

Router kinds: "normal" (no bias), "bias_normal" (bias_e ~ N(0, variance 0.5)), "zipf"
(bias_e = ln p_e with p_e proportional to (e+1)^-1.2, expert 0 most popular).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Optional

import numpy as np
import torch

from .configs import FMT_FP8, FMT_MXFP8, FMT_NVFP4, FMT_W4A4, TailConfig

__all__ = ["make_activations", "make_weights", "make_inputs", "make_projection_weights",
           "fp8_block_quantize", "mx_quantize", "nvfp4_quantize", "expert_load"]


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> torch.Tensor:
    t = torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32))
    if std != 1.0:
        t.mul_(std)
    return t


# ---------------------------------------------------------------- offline weight formats

def fp8_block_quantize(w: torch.Tensor):
    """[R, C] fp32 -> (e4m3 codes uint8 [R, C], fp32 scales [R/128, C/128]).

    One scale per 128x128 block: amax/448 (1 for an all-zero block); codes are the
    clamped quotient cast by PyTorch (round to nearest even)."""
    R, C = w.shape
    b = w.reshape(R // 128, 128, C // 128, 128)
    amax = b.abs().amax(dim=(1, 3))
    s = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
    v = (b / s[:, None, :, None]).clamp_(-448.0, 448.0)
    q = v.to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, C)
    return q, s.contiguous()


def mx_quantize(w: torch.Tensor):
    """[R, C] fp32 -> (e4m3 codes uint8 [R, C], UE8M0 scale bytes uint8 [R, C/32]).

    One power-of-two scale per 32 consecutive K-elements of a row: 2^(floor(log2 amax) - 8)
    (1 for an all-zero block), the byte holding exponent + 127; codes are the clamped
    quotient cast by PyTorch (round to nearest even)."""
    R, C = w.shape
    b = w.reshape(R, C // 32, 32)
    amax = b.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)
    e = torch.where(amax > 0, ex - 9, torch.zeros_like(ex)).clamp_(-127, 127)
    v = (b / torch.ldexp(torch.ones_like(amax), e)[..., None]).clamp_(-448.0, 448.0)
    q = v.to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, C)
    return q, (e + 127).to(torch.uint8).contiguous()


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Nearest e2m1 code (ties to the even code) of fp32 values already scaled to +-6."""
    a = v.abs()
    code = ((a > 0.25).to(torch.uint8) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5)
            + (a >= 3.5) + (a > 5.0)).to(torch.uint8)
    sign = ((v < 0) & (code > 0)).to(torch.uint8) << 3
    return code | sign


def nvfp4_quantize(w: torch.Tensor):
    """[R, C] fp32 -> (packed e2m1 uint8 [R, C/2], e4m3 block scales uint8 [R, C/16],
    fp32 per-matrix scale).  Two codes per byte, the even K index in the low nibble."""
    R, C = w.shape
    amax = float(w.abs().max())
    g = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    blk = w.reshape(R, C // 16, 16)
    bamax = blk.abs().amax(dim=-1)
    sbv = (bamax / 6.0 / float(g)).clamp_(max=448.0)
    sb = sbv.to(torch.float8_e4m3fn)
    scale = sb.to(torch.float32) * float(g)
    safe = torch.where(scale == 0, torch.ones_like(scale), scale)
    v = (blk / safe[..., None]).clamp_(-6.0, 6.0)
    v = torch.where((scale == 0)[..., None], torch.zeros_like(v), v)
    codes = _e2m1_codes(v).reshape(R, C)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed.contiguous(), sb.view(torch.uint8).contiguous(), float(g)


# ---------------------------------------------------------------- draws

def _router_bias(cfg: TailConfig, rng: np.random.Generator) -> Optional[np.ndarray]:
    if cfg.router == "normal":
        return None
    if cfg.router == "bias_normal":
        return (rng.standard_normal(cfg.E) * math.sqrt(0.5)).astype(np.float32)
    if cfg.router == "zipf":
        p = (np.arange(cfg.E, dtype=np.float64) + 1.0) ** -1.2
        p /= p.sum()
        return np.log(p).astype(np.float32)
    raise ValueError(f"unknown router kind {cfg.router!r}")


def make_activations(cfg: TailConfig, M: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Token inputs: x [M,H] bf16, z [M,L] bf16, logits [M,E] fp32 (bias included)."""
    M = cfg.M if M is None else M
    rng = _rng(cfg.seed, 0)
    x = _normal(rng, (M, cfg.H)).to(torch.bfloat16)
    z = _normal(rng, (M, cfg.L)).to(torch.bfloat16)
    logits = rng.standard_normal(size=(M, cfg.E), dtype=np.float32)
    bias = _router_bias(cfg, rng)
    if bias is not None:
        logits = (logits + bias[None, :]).astype(np.float32)
    return {"x": x, "z": z, "logits": torch.from_numpy(logits)}


def make_weights(cfg: TailConfig) -> Dict[str, torch.Tensor]:
    """All weights of one tail layer in their stored formats (CPU tensors)."""
    rng = _rng(cfg.seed, 1)
    E, H, L, I, Is = cfg.E, cfg.H, cfg.L, cfg.I, cfg.Is
    w: Dict[str, torch.Tensor] = {}
    w["gamma"] = torch.from_numpy(rng.uniform(0.5, 1.5, size=L).astype(np.float32)).to(
        torch.bfloat16)
    if cfg.routed_fmt == FMT_FP8:
        w13_q = torch.empty((E, 2 * I, L), dtype=torch.uint8)
        w13_s = torch.empty((E, 2 * I // 128, L // 128), dtype=torch.float32)
        for e in range(E):
            w13_q[e], w13_s[e] = fp8_block_quantize(_normal(rng, (2 * I, L), 1 / math.sqrt(L)))
        w2_q = torch.empty((E, L, I), dtype=torch.uint8)
        w2_s = torch.empty((E, L // 128, I // 128), dtype=torch.float32)
        for e in range(E):
            w2_q[e], w2_s[e] = fp8_block_quantize(_normal(rng, (L, I), 1 / math.sqrt(I)))
        w.update(w13_q=w13_q, w13_s=w13_s, w2_q=w2_q, w2_s=w2_s)
    elif cfg.routed_fmt == FMT_MXFP8:
        w13_q = torch.empty((E, 2 * I, L), dtype=torch.uint8)
        w13_sx = torch.empty((E, 2 * I, L // 32), dtype=torch.uint8)
        for e in range(E):
            w13_q[e], w13_sx[e] = mx_quantize(_normal(rng, (2 * I, L), 1 / math.sqrt(L)))
        w2_q = torch.empty((E, L, I), dtype=torch.uint8)
        w2_sx = torch.empty((E, L, I // 32), dtype=torch.uint8)
        for e in range(E):
            w2_q[e], w2_sx[e] = mx_quantize(_normal(rng, (L, I), 1 / math.sqrt(I)))
        w.update(w13_q=w13_q, w13_sx=w13_sx, w2_q=w2_q, w2_sx=w2_sx)
    elif cfg.routed_fmt in (FMT_NVFP4, FMT_W4A4):  # the same NVFP4 weights
        w13_q = torch.empty((E, 2 * I, L // 2), dtype=torch.uint8)
        w13_sb = torch.empty((E, 2 * I, L // 16), dtype=torch.uint8)
        w13_g = torch.empty(E, dtype=torch.float32)
        for e in range(E):
            w13_q[e], w13_sb[e], w13_g[e] = nvfp4_quantize(
                _normal(rng, (2 * I, L), 1 / math.sqrt(L)))
        w2_q = torch.empty((E, L, I // 2), dtype=torch.uint8)
        w2_sb = torch.empty((E, L, I // 16), dtype=torch.uint8)
        w2_g = torch.empty(E, dtype=torch.float32)
        for e in range(E):
            w2_q[e], w2_sb[e], w2_g[e] = nvfp4_quantize(_normal(rng, (L, I), 1 / math.sqrt(I)))
        w.update(w13_q=w13_q, w13_sb=w13_sb, w13_g=w13_g, w2_q=w2_q, w2_sb=w2_sb, w2_g=w2_g)
    else:
        raise ValueError(f"unknown routed format {cfg.routed_fmt!r}")
    w["ws13"] = _normal(rng, (2 * Is, H), 1 / math.sqrt(H)).to(torch.bfloat16)
    w["ws2"] = _normal(rng, (H, Is), 1 / math.sqrt(Is)).to(torch.bfloat16)
    w["w_up"] = _normal(rng, (H, L), 1 / math.sqrt(L)).to(torch.bfloat16)
    return w


def make_projection_weights(cfg: TailConfig) -> Dict[str, torch.Tensor]:
    """Weights of the step before the tail (hidden state -> latent input and router
    logits), drawn from their own stream ``default_rng([seed, 2])`` so that the tail's own
    draws are unchanged: w_lat [L, H] and w_gate [E, H], both ~ N(0, 1/H) stored as bf16."""
    rng = _rng(cfg.seed, 2)
    w_lat = _normal(rng, (cfg.L, cfg.H), 1 / math.sqrt(cfg.H)).to(torch.bfloat16)
    w_gate = _normal(rng, (cfg.E, cfg.H), 1 / math.sqrt(cfg.H)).to(torch.bfloat16)
    return {"w_lat": w_lat, "w_gate": w_gate}


def make_inputs(cfg: TailConfig, M: Optional[int] = None):
    """(activations, weights) for one workload."""
    return make_activations(cfg, M), make_weights(cfg)


def expert_load(logits: torch.Tensor, topk: int) -> np.ndarray:
    """Tokens per expert under plain top-k selection of the logits (a workload statistic
    used to check the skew recipe; ties do not matter for a histogram of random floats)."""
    ids = torch.topk(logits, topk, dim=1).indices.reshape(-1)
    return torch.bincount(ids, minlength=logits.shape[1]).numpy()

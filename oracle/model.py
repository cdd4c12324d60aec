"""Plain CPU float64 oracle of the latent-MoE layer tail.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
timing leg of ``bench.py`` may import this package.  It shares no code with the CUDA
path; the two meet only through the seeded inputs.

What it computes, step by step (sources are the four pages on the Kimi K3 latent MoE:
vLLM "Fuse BF16 shared experts into latent MegaMoE tail" (Summary), DeepGEMM PR 416
"Fuse and publish Kimi K3's BF16 shared expert" (Summary), the tokenspeed recipe
"Kimi-K3 DEP16 with sharded shared experts" (Communication and validation) and tokenspeed
PR 1062 "MNNVL CuTe-DSL finalize tail" (commit notes and Summary)):

1. Route: per token, the k largest router logits (ties: lower expert index first), weights
   = softmax over the selected k logits (so they sum to 1).
2. Quantise the latent input z per token per 128 columns to e4m3 with an fp32 scale
   amax/448 (scale 1 for an all-zero group), quotient and scale in fp32, round to nearest
   even, saturating.
3. Routed experts in the 3584-wide latent space: h = deq(zq) deq(W13_e)^T, gate = first I
   rows of W13_e, up = next I; a = silu(gate) * up; a is quantised per 128 like step 2
   (from float32(a)); y = deq(aq) deq(W2_e)^T.
4. Combine ("finalize"): r = sum_j w_j y_j (top-k weighted sum).
5. RMSNorm of r (eps, weight gamma), then the 3584 -> 7168 up-projection.
6. Shared expert on the 7168-wide hidden state: gate/up -> SwiGLU -> down.
7. out = up-projection + shared output (the oracle rounds nothing here; the tail emits
   bf16).

Format variants of steps 2 and 3 (DeepGEMM PR 416, Summary: the FP8/FP4 MegaMoE path):
MXFP8 quantises activations per 32 with power-of-two scales (OCP Microscaling rule), and
the FP4 x FP4 format quantises them to NVFP4 (e2m1, one e4m3 scale per 16) like its
weights.

Every product and sum runs in float64 on exactly dequantised weights.
"""
from __future__ import annotations

from typing import Dict, Iterable, Optional

import numpy as np

from .codecs import e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode, unpack_e2m1

__all__ = ["route", "permutation", "quant_per128", "silu", "dequant_fp8_blocks",
           "dequant_nvfp4", "rmsnorm", "swiglu_mlp", "tail", "to_f64", "latent_inputs",
           "bf16_round", "quant_mx", "dequant_mx", "quant_nvfp4", "dequant_nvfp4_act"]


def to_f64(t) -> np.ndarray:
    """torch tensor (any float dtype) or array -> float64 numpy array (exact)."""
    if hasattr(t, "detach"):
        import torch
        return t.detach().to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def _rows_f64(t, rows) -> np.ndarray:
    if hasattr(t, "detach"):
        import torch
        return to_f64(t[torch.as_tensor(rows, dtype=torch.long)])
    return np.asarray(t, dtype=np.float64)[rows]


def _np(t) -> np.ndarray:
    return t.detach().numpy() if hasattr(t, "detach") else np.asarray(t)


# ---------------------------------------------------------------- step 0: inputs from x

def bf16_round(v) -> np.ndarray:
    """float64 -> nearest bfloat16 value (ties to even), returned as float64."""
    import torch
    return torch.from_numpy(np.asarray(v, dtype=np.float64)).to(torch.bfloat16).to(
        torch.float64).numpy()


def latent_inputs(x, w_lat, w_gate):
    """The step before the tail (tokenspeed PR 1062, commit notes: the model's latent input
    projections feed the latent MoE).  Reading: both come from the hidden state x; the
    latent input is z = x W_lat^T (H -> L), stored as bf16 (the tail's z is a bf16 tensor),
    and the router logits are x W_gate^T kept in full precision.  Returns (z as float64
    holding bf16 values [M, L], logits float64 [M, E])."""
    xv = to_f64(x)
    z = bf16_round(xv @ to_f64(w_lat).T)
    logits = xv @ to_f64(w_gate).T
    return z, logits


# ---------------------------------------------------------------- step 1: route

def route(logits, k: int):
    """Top-k of each row (descending logit, ties to the lower index) and the softmax of
    the selected logits.  Returns (ids int32 [M,k], w float64 [M,k])."""
    lg = np.asarray(_np(logits), dtype=np.float32).astype(np.float64)
    order = np.argsort(-lg, axis=1, kind="stable")
    ids = order[:, :k]
    sel = np.take_along_axis(lg, ids, axis=1)
    ex = np.exp(sel - sel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w


def permutation(ids, E: int):
    """Stable grouping of the (token, choice) pairs by expert.

    Pair i = t*k + j.  p runs over pairs sorted by expert, pairs of one expert in
    ascending i (hence ascending token).  Returns cnt[E], off[E+1], gidx[M*k] (token of
    pair p), slot[M*k] (= i of pair p), pos[M,k] (p of pair (t, j))."""
    ids = np.asarray(ids)
    M, k = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")
    cnt = np.bincount(flat, minlength=E).astype(np.int32)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(cnt)
    slot = order.astype(np.int32)
    gidx = (order // k).astype(np.int32)
    pos = np.empty(M * k, dtype=np.int32)
    pos[order] = np.arange(M * k, dtype=np.int32)
    return cnt, off, gidx, slot, pos.reshape(M, k)


# ---------------------------------------------------------------- step 2: act quant

def quant_per128(v32):
    """Per row, per 128 columns: s = fp32(amax)/448 (1 if amax == 0); q = e4m3(v/s) with
    the quotient in fp32.  Returns (codes uint8 [n,C], scales float32 [n,C/128])."""
    v = np.asarray(v32, dtype=np.float32)
    n, C = v.shape
    g = v.reshape(n, C // 128, 128)
    amax = np.abs(g).max(axis=-1)
    s = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0)).astype(np.float32)
    quot = (g / s[..., None]).astype(np.float32)
    q = e4m3_encode(quot).reshape(n, C)
    return q, s


def quant_mx(v32):
    """MX e4m3 quantisation (OCP Microscaling formats v1.0, e4m3 elements): per row, per 32
    columns, one shared power-of-two scale X = 2^(floor(log2(amax)) - 8) (8 = the largest
    e4m3 exponent), stored as an UE8M0 byte (exponent + 127, clamped to 0..254); elements
    q = e4m3(v / X), nearest even, saturating at +-448.  An all-zero block takes X = 1.
    Returns (codes uint8 [n,C], scale bytes uint8 [n,C/32])."""
    v = np.asarray(v32, dtype=np.float32)
    n, C = v.shape
    g = v.reshape(n, C // 32, 32)
    amax = np.abs(g).max(axis=-1).astype(np.float64)
    _, ex = np.frexp(amax)                   # amax = m * 2^ex, 0.5 <= m < 1
    e = np.where(amax > 0, ex - 1 - 8, 0)    # floor(log2(amax)) - 8
    e = np.clip(e, -127, 127)
    quot = (g.astype(np.float64) / np.ldexp(1.0, e)[..., None]).astype(np.float32)
    q = e4m3_encode(quot).reshape(n, C)
    return q, (e + 127).astype(np.uint8)


def dequant_mx(q, sb) -> np.ndarray:
    """MX e4m3 codes [n,C] with UE8M0 bytes [n,C/32] -> float64 (exact)."""
    q = np.asarray(q)
    n, C = q.shape
    scale = np.ldexp(1.0, np.asarray(sb, dtype=np.int64) - 127)
    return (e4m3_decode(q).reshape(n, C // 32, 32) * scale[..., None]).reshape(n, C)


def quant_nvfp4(v32):
    """NVFP4 activation quantisation (e2m1 elements, one e4m3 scale per 16, no tensor-wide
    scale): per row, per 16 columns, s = e4m3(fp32(amax / 6)) (nearest even, saturating
    at 448); elements q = e2m1(fp32(v / s)), nearest even, saturating at 6, no negative
    zero.  A block whose scale is zero (amax below the smallest e4m3 step) has all codes 0.
    Returns (codes uint8 [n,C], one 4-bit code per element; scale bytes uint8 [n,C/16])."""
    v = np.asarray(v32, dtype=np.float32)
    n, C = v.shape
    g = v.reshape(n, C // 16, 16)
    amax = np.abs(g).max(axis=-1)
    sb = e4m3_encode((amax / np.float32(6.0)).astype(np.float32))
    s = e4m3_decode(sb).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s)
    quot = (g / safe[..., None]).astype(np.float32)
    q = np.where((s == 0)[..., None], np.uint8(0), e2m1_encode(quot))
    return q.reshape(n, C).astype(np.uint8), sb


def dequant_nvfp4_act(q, sb) -> np.ndarray:
    """e2m1 codes [n,C] (one per element) with e4m3 scale bytes [n,C/16] -> float64."""
    q = np.asarray(q)
    n, C = q.shape
    return (e2m1_decode(q).reshape(n, C // 16, 16)
            * e4m3_decode(sb)[..., None]).reshape(n, C)


def dequant_act(q, s) -> np.ndarray:
    q = np.asarray(q)
    n, C = q.shape
    return (e4m3_decode(q).reshape(n, C // 128, 128)
            * np.asarray(s, dtype=np.float64)[..., None]).reshape(n, C)


# ---------------------------------------------------------------- weights

def dequant_fp8_blocks(q, s) -> np.ndarray:
    """e4m3 codes [R,C] with fp32 scales [R/128,C/128] -> float64 [R,C]."""
    q = _np(q)
    R, C = q.shape
    v = e4m3_decode(q).reshape(R // 128, 128, C // 128, 128)
    return (v * np.asarray(_np(s), dtype=np.float64)[:, None, :, None]).reshape(R, C)


def dequant_nvfp4(packed, sb, g) -> np.ndarray:
    """packed e2m1 [R,C/2], e4m3 block scales [R,C/16], fp32 matrix scale -> float64."""
    codes = unpack_e2m1(_np(packed))
    R, C = codes.shape
    vals = e2m1_decode(codes).reshape(R, C // 16, 16)
    scale = e4m3_decode(_np(sb)) * float(g)
    return (vals * scale[..., None]).reshape(R, C)


# ---------------------------------------------------------------- math pieces

def silu(v):
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def rmsnorm(r, gamma, eps: float):
    """r / sqrt(mean(r^2) + eps) * gamma, per row."""
    r = np.asarray(r, dtype=np.float64)
    return r / np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + eps) * gamma


def swiglu_mlp(x, w13, w2):
    """SwiGLU MLP: gate = first half of w13's rows, up = second half."""
    inter = w13.shape[0] // 2
    h = x @ w13.T
    return (silu(h[:, :inter]) * h[:, inter:]) @ w2.T


# ---------------------------------------------------------------- the tail

def _expert_weights(w: Dict, fmt: str, e: int):
    if fmt == "fp8":
        return (dequant_fp8_blocks(w["w13_q"][e], w["w13_s"][e]),
                dequant_fp8_blocks(w["w2_q"][e], w["w2_s"][e]))
    if fmt == "mxfp8":
        return (dequant_mx(_np(w["w13_q"][e]), _np(w["w13_sx"][e])),
                dequant_mx(_np(w["w2_q"][e]), _np(w["w2_sx"][e])))
    # "nvfp4" and "nvfp4_w4a4" share the NVFP4 weight format
    return (dequant_nvfp4(w["w13_q"][e], w["w13_sb"][e], float(w["w13_g"][e])),
            dequant_nvfp4(w["w2_q"][e], w["w2_sb"][e], float(w["w2_g"][e])))


def tail(act: Dict, w: Dict, cfg, tokens: Optional[Iterable[int]] = None) -> Dict:
    """Run the whole tail.  ``tokens`` limits the per-token work to a subset (each token's
    output depends on that token alone); routing and the permutation always cover every
    token.  Returns every intermediate, indexed by the selected tokens' order."""
    k, E, I = cfg.topk, cfg.E, cfg.I
    logits = act["logits"]
    M = logits.shape[0]
    ids, wts = route(logits, k)
    cnt, off, gidx, slot, pos = permutation(ids, E)
    tok = np.arange(M) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    n = len(tok)

    # activation quantiser: fp32 amax/448 per 128 columns, MX (power-of-two per 32), or
    # NVFP4 (e2m1 with an e4m3 scale per 16) for the FP4 x FP4 format
    mx = cfg.routed_fmt == "mxfp8"
    a4 = cfg.routed_fmt == "nvfp4_w4a4"
    quant, deq, G = ((quant_mx, dequant_mx, 32) if mx else
                     (quant_nvfp4, dequant_nvfp4_act, 16) if a4 else
                     (quant_per128, dequant_act, 128))
    z = _rows_f64(act["z"], tok)
    zq, zs = quant(z.astype(np.float32))
    zdq = deq(zq, zs)

    # Routed experts, one expert at a time (bounded memory).
    r = np.zeros((n, cfg.L))
    aq = np.zeros((n, k, I), dtype=np.uint8)
    as_ = np.zeros((n, k, I // G), dtype=np.uint8 if (mx or a4) else np.float32)
    sel_ids = ids[tok]
    for e in np.unique(sel_ids):
        rows, js = np.nonzero(sel_ids == e)
        w13, w2 = _expert_weights(w, cfg.routed_fmt, int(e))
        h = zdq[rows] @ w13.T
        a = silu(h[:, :I]) * h[:, I:]
        q, s = quant(a.astype(np.float32))
        aq[rows, js], as_[rows, js] = q, s
        y = deq(q, s) @ w2.T
        np.add.at(r, rows, wts[tok][rows, js][:, None] * y)

    gamma = to_f64(w["gamma"])
    nrm = rmsnorm(r, gamma, cfg.eps)
    up = nrm @ to_f64(w["w_up"]).T

    x = _rows_f64(act["x"], tok)
    ws13 = to_f64(w["ws13"])
    hs = x @ ws13.T
    a_s = silu(hs[:, :cfg.Is]) * hs[:, cfg.Is:]
    s_out = a_s @ to_f64(w["ws2"]).T

    return {
        "tokens": tok, "ids": ids, "w": wts, "cnt": cnt, "off": off, "gidx": gidx,
        "slot": slot, "pos": pos, "zq": zq, "zs": zs, "aq": aq, "as": as_, "r": r,
        "n": nrm, "up": up, "a_s": a_s, "s": s_out, "out": up + s_out,
    }
